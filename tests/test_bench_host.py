"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes and
flops behind the roofline, the ncu traffic lookup that is only trusted while
the kernel source is unchanged since the capture, and the peaks file."""

import json
import os
import shutil

import pytest

import bench


def test_algorithmic_units():
    # Fused norm+quant per row: q 3072 + kv 1024 read; codes 1536 + 12 fp32
    # scales + kv 1024 written.  Unfused: norm (4096 in, 4096 out) and two
    # group quants (3072 in, 1536 + 48 out each).
    assert bench.NQ_BYTES_PER_ROW == 3072 + 1024 + 1536 + 48 + 1024 == 6704
    assert bench.UNFUSED_BYTES_PER_ROW == 17504
    assert bench.NQ_BYTES_PER_CALL == 4096
    assert bench.gemm_flops(8192) == 2 * 8192 * (24576 + 4096) * 1536
    assert abs(bench.gemm_flops(8192) / 1e9 - 721.6) < 0.1


def test_captured_traffic_matches_committed_sources():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, r in rec.items():
        got = bench.captured_traffic(key)
        assert got == r["dram_bytes_per_launch"], key
    assert bench.captured_traffic("no_such_kernel") is None


def test_captured_traffic_is_dropped_when_the_source_changes(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    (root / "gemm_dsnq_dual_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"), root / "profiles" / "traffic.json")
    src = os.path.join(bench.ROOT, "gemm_dsnq_dual_gb300", "csrc", "gemm_fp8.cu")
    dst = root / "gemm_dsnq_dual_gb300" / "csrc" / "gemm_fp8.cu"
    shutil.copy(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.captured_traffic("gemm_dual_M8192") is not None
    dst.write_bytes(dst.read_bytes() + b"\n// changed\n")
    assert bench.captured_traffic("gemm_dual_M8192") is None


def test_peaks_come_from_the_measured_file():
    hbm, bf16, sustained, source = bench.load_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        d = json.load(open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")))
        assert (hbm, bf16, source) == (d["hbm_gbs"], d["bf16_tflops"], "measured")
    else:
        assert source == "fallback"


@pytest.mark.parametrize("world", [1, 2, 8])
def test_whole_job_value_counts_every_rank(world):
    # TFLOP/s of all ranks' work over the slowest rank's step time.
    assert bench.whole_job_value(world, 1e12, 2.0) == pytest.approx(world * 1e12 / 2e-3 / 1e12)
