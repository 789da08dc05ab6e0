"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes and
flops behind the roofline, the ncu traffic lookup that is only trusted while
the kernel source is unchanged since the capture, and the peaks file."""

import json
import os

import pytest

import bench


@pytest.mark.parametrize("M", [1024, 2048, 8192, 32768])
def test_graph_sets_keep_every_call_cold(M):
    """A graph cycling over the sets revisits one only after more than L2's
    worth (160 MiB) of the others."""
    per_set = M * bench.NQ_BYTES_PER_ROW
    n = bench.graph_sets(per_set)
    assert n >= 2 and (n - 1) * per_set > 160 * 2 ** 20
    assert (n - 2) * per_set <= 160 * 2 ** 20 or n == 2      # no more sets than that needs


def test_algorithmic_units():
    # Fused norm+quant per row: q 3072 + kv 1024 read; codes 1536 + 12 fp32
    # scales + kv 1024 written.  Unfused: norm (4096 in, 4096 out) and two
    # group quants (3072 in, 1536 + 48 out each).
    assert bench.NQ_BYTES_PER_ROW == 3072 + 1024 + 1536 + 48 + 1024 == 6704
    assert bench.UNFUSED_BYTES_PER_ROW == 17504
    assert bench.NQ_BYTES_PER_CALL == 4096
    assert bench.gemm_flops(8192) == 2 * 8192 * (24576 + 4096) * 1536
    assert abs(bench.gemm_flops(8192) / 1e9 - 721.6) < 0.1


def test_committed_traffic_records_are_well_formed():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, r in rec.items():
        assert r["dram_bytes_per_launch"] > 0, key
        assert os.path.exists(os.path.join(bench.ROOT, "gemm_dsnq_dual_gb300", "csrc", r["source"])), key
        assert len(r["source_sha256_16"]) == 16, key
    assert bench.captured_traffic("no_such_kernel") is None


def test_captured_traffic_only_while_the_source_is_unchanged(tmp_path, monkeypatch):
    """A record is used only while the hash of the kernel source it names
    still matches the source the capture was taken from."""
    import hashlib
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    (root / "gemm_dsnq_dual_gb300" / "csrc").mkdir(parents=True)
    src = root / "gemm_dsnq_dual_gb300" / "csrc" / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    json.dump({"k_M1": {"dram_bytes_per_launch": 1234, "source": "k.cu", "source_sha256_16": h}},
              open(root / "profiles" / "traffic.json", "w"))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.captured_traffic("k_M1") == 1234
    src.write_bytes(src.read_bytes() + b"// changed\n")
    assert bench.captured_traffic("k_M1") is None


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


def test_headline_keeps_the_metric_numbers():
    """The compact summary printed last on the bench line carries the
    figures the metric is quoted on."""
    line = {"roofline": {"achieved": 2000.0, "frac": 0.51}, "roofline_norm_quant": {"frac": 0.4},
            "norm_quant_us_at_M1": 2.4,
            "norm_quant_sweep": {"8192": {"fused_graph_frac_hbm": 0.52, "speedup_vs_unfused": 2.5}, "note": "x"},
            "decode_step_us_at_M1": {"overlap": 13.0, "one_launch": 12.3},
            "gemm_sweep": {"1": {"graph_us": 10.8, "graph_frac_hbm": 0.6}, "1024": {"tflops": 1600.0},
                           "32768_long_context_attn": {"tflops": 2000.0, "frac_fp8": 0.52}},
            "decode_sweep": {"1": {"row_us": 2.5, "col_us": 2.5}, "note": "x"},
            "single_latent_norm_quant": {"1": {"graph_us": 2.2}, "8192": {"graph_frac_hbm": 0.6}, "note": "x"},
            "cpu_baseline": {"cores": 16, "value": 0.1, "single_thread": {"value": 0.02}}}
    h = bench.headline(line)
    assert h["norm_quant_us_at_M1"] == 2.4
    assert h["norm_quant_graph_frac_hbm"] == {"8192": 0.52}
    assert h["gemm_attn_M32768_frac_fp8"] == 0.52 and h["gemm_dual_M8192_frac_fp8"] == 0.51
    assert h["norm_quant_decode_us"] == {"1": [2.5, 2.5]}
    assert h["decode_step_us_at_M1"] == 13.0 and h["decode_step_us_at_M1_one_launch"] == 12.3
    assert h["single_latent_us_at_M1"] == 2.2 and h["single_latent_graph_frac_hbm"] == {"8192": 0.6}
    assert h["cpu_oracle_tflops"] == {"cores": 16, "all": 0.1, "one_thread": 0.02}


def test_both_arms_describe_the_same_workload():
    assert bench.step_config(8192, 1) == bench.step_config(8192, 1)
    assert bench.step_config(8192, 1)["M"] == 8192


def test_cpu_baseline_times_the_oracle_on_one_and_all_cores():
    """The oracle runs in child processes (one thread, then all cores) on a
    small sample here; the line reports both with their core counts."""
    r = bench.cpu_baseline(8)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s"
    assert r["cores"] == bench.host_cores() >= 1
    assert r["single_thread"]["cores"] == 1
    assert r["value"] > 0 and r["single_thread"]["value"] > 0
