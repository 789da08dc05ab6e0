"""Benchmark of the decode-step MLA latent pre-projection on GB300.

One step = the whole hot path over one batch of M token rows:
  fused dual RMSNorm + per-1x128 FP8 quant (q [M,1536], kv [M,512] bf16)
  -> block-scaled FP8 GEMM for both consumers in one launch
     (attention wq_b N=24576 and indexer wq_b N=4096, K=1536, bf16 out).
Default workload: the full-path configuration at M=8192 tokens, synthetic
inputs (N(0,1) latents, U(0.5,1.5) gammas, N(0,0.02) weights quantized per
128x128 block), resident in HBM.  L2 is flushed (256 MiB written, another
256 MiB read) before every timed step; each step is timed with CUDA events
on the launch stream.

The JSON line also reports, measured in the same run:
  * per-kernel times and roofline fractions (GEMM vs the FP8 tensor peak,
    norm+quant vs HBM bandwidth), against MEASURED_PEAKS.json when present;
  * the norm+quant latency at M=1 (decode), from a CUDA graph of 100 calls on
    100 cold rows (with launch overlap on and off), and its GB/s at
    M=1024/8192/32768;
  * one decode step at M=1 (norm+quant, then the dual GEMM over cold
    weights): two launches with and without launch overlap, the one-launch
    call, and the dual GEMM on a bf16 row quantized inside the GEMM or by the
    quant kernel first;
  * the dual GEMM alone over decode and larger batch sizes;
  * the unfused three-kernel sequence (dual RMSNorm to bf16, then the per-1x128
    quant twice) on the same GPU at the same M;
  * e2e: the same step through the public API with pinned host buffers
    (inputs copied in, both projections and kv copied out, inside the timer;
    consecutive steps overlap on three streams, as a serving loop runs them);
  * cpu_baseline: the fp64 CPU oracle timed on the whole M=8192 workload.

`--impl reference` times the CPU oracle alone on the same metric (bounded
samples of rows and output columns so the run ends within minutes).
Multi-GPU: rows are independent, so each rank runs its own batch (weak
scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

KQ, KKV, N_ATTN, N_IDX = 1536, 512, 24576, 4096
# Back-to-back decode calls per CUDA graph (the steady state of a decode loop,
# which runs every layer's kernels one after another).
DECODE_GRAPH_CALLS = 100
# Norm+quant at M >= 1024: calls per CUDA graph (at least), cycling over
# distinct input/output sets; a set is revisited only after more than L2's
# worth of other sets (cold every time).
NQ_GRAPH_CALLS = 100
METRIC = "norm+quant HBM GB/s (% of peak) & µs at M=1; block-scaled FP8 GEMM TFLOPS"
NQ_BYTES_PER_ROW = 2 * KQ + 2 * KKV + KQ + 4 * (KQ // 128) + 2 * KKV   # 6704
NQ_BYTES_PER_CALL = 2 * (KQ + KKV)                                      # gammas
UNFUSED_BYTES_PER_ROW = (4096 + 4096) + 2 * (3072 + 1584)               # 17504


def step_config(M: int, world: int) -> dict:
    """The workload one step processes (the same for both arms)."""
    return {"workload": f"full path: fused dual RMSNorm + per-1x128 FP8 quant of q[{M},1536]/kv[{M},512] "
                        f"-> dual block-scaled FP8 GEMM (wq_b N=24576 + indexer wq_b N=4096, K=1536)",
            "M": M, "Kq": KQ, "Kkv": KKV, "N": [N_ATTN, N_IDX], "scale_layout": "column-major",
            "l2": "flushed before every timed step (256 MiB write + 256 MiB read)",
            "parallelism": f"dp{world} (independent token batches, no collective)"}


def gemm_flops(M: int) -> float:
    return 2.0 * M * (N_ATTN + N_IDX) * KQ


def captured_traffic(key: str, field: str = "dram_bytes_per_launch"):
    """DRAM bytes per launch (read + write), or another `field` of the record,
    from the committed ncu summary; None when the kernel's source has changed
    since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(key)
    if not rec:
        return None
    src = os.path.join(ROOT, "gemm_dsnq_dual_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec.get(field)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx = float(parts[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        busy = [s for s in sm if mx is None or s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- GPU arm

class L2Flush:
    """Evicts the L2 (129 MB on GB300) between timed steps: writes one 256 MiB
    buffer, then reads a second one, so the dirty lines of the write are
    written back during the flush and not during the next timed kernel."""

    def __init__(self, torch, dev):
        n = 256 * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()

def run_ours(args, rank, world):
    import torch
    import gemm_dsnq_dual_gb300 as dsnq
    from gemm_dsnq_dual_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    M = args.M
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = load_peaks()
    fp8_peak = 2.0 * bf16_tf            # FP8 dense = 2x bf16 dense (nominal ratio)

    # ---- inputs and weights, resident in HBM (weights quantized on the GPU at load time)
    lat = inputs.full_path_batch(M, seed=rank_seed(rank))
    q, kv = lat.q.to(dev), lat.kv.to(dev)
    gq, gkv = lat.gamma_q.to(dev), lat.gamma_kv.to(dev)
    wa, swa = dsnq.quantize_weight_block128(inputs.weight(N_ATTN, KQ, seed=0, salt=1).to(dev))
    wi, swi = dsnq.quantize_weight_block128(inputs.weight(N_IDX, KQ, seed=0, salt=2).to(dev))
    q_fp8 = torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev)
    q_scale = dsnq.empty_scales(M, KQ // 128, "col", dev)
    kv_out = torch.empty(M, KKV, dtype=torch.bfloat16, device=dev)
    out_a = torch.empty(M, N_ATTN, dtype=torch.bfloat16, device=dev)
    out_i = torch.empty(M, N_IDX, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()

    def norm_quant():
        dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="col",
                                            q_out=q_fp8, q_scale=q_scale, kv_out=kv_out)

    def gemm():
        dsnq.block_scaled_fp8_gemm_dual(q_fp8, q_scale, wa, swa, wi, swi, out1=out_a, out2=out_i)

    def step():
        norm_quant()
        gemm()

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        for i in range(K):
            flush()                      # cold L2 for every step (outside the events)
            ev[i][0].record(stream)
            norm_quant()
            ev[i][1].record(stream)
            gemm()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    nq_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    gm_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = sum(nq_ms) / K + sum(gm_ms) / K
    step_ms_max = allreduce_max(step_ms, world, dev)
    clocks = clk.summary()

    # ---- side measurements (rank 0 only; not part of the timed region)
    extra = {}
    if rank == 0:
        extra = side_measurements(torch, dsnq, inputs, dev, flush, hbm_gbs, args, fp8_peak)
        extra["e2e"] = e2e_measurement(torch, dsnq, lat, dev, (wa, swa, wi, swi), args, M)
    if rank != 0:
        return

    nq_avg, gm_avg = sum(nq_ms) / K, sum(gm_ms) / K
    gemm_tflops = gemm_flops(M) / (gm_avg * 1e-3) / 1e12
    nq_gbs = (M * NQ_BYTES_PER_ROW + NQ_BYTES_PER_CALL) / (nq_avg * 1e-3) / 1e9
    value = whole_job_value(world, gemm_flops(M), step_ms_max)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3xe4m3->f32 (GEMM); bf16->f32->e4m3/bf16 (norm+quant)",
        "data": "synthetic",
        "config": step_config(M, world),
        "gpu_launches": 2 * K,
        "kernels": {
            "norm_quant_us": round(nq_avg * 1e3, 3),
            "norm_quant_gbs": round(nq_gbs, 1),
            "gemm_dual_us": round(gm_avg * 1e3, 3),
            "gemm_dual_tflops": round(gemm_tflops, 1),
        },
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": captured_traffic(f"gemm_dual_M{M}"),
                     "tensor_pipe_active_pct": captured_traffic(f"gemm_dual_M{M}", "tensor_pipe_active_pct"),
                     "algorithmic_bytes": int(M * (KQ + 4 * KQ // 128) + (N_ATTN + N_IDX) * KQ
                                              + 2 * M * (N_ATTN + N_IDX)),
                     "kernel": ("pair_gemm_kernel" if M >= 256 else "block_scaled_gemm_kernel") + " (one launch, both consumers)",
                     "peak_source": f"{peak_src}: FP8 = 2 x bf16 dense burst ({bf16_tf} TFLOP/s)"},
        "roofline_norm_quant": {"bound": "hbm", "achieved": round(nq_gbs, 1), "peak": hbm_gbs,
                                "unit": "GB/s", "frac": round(nq_gbs / hbm_gbs, 4),
                                "traffic": captured_traffic(f"norm_quant_M{M}"),
                                "algorithmic_bytes": M * NQ_BYTES_PER_ROW + NQ_BYTES_PER_CALL,
                                "peak_source": peak_src},
        "wall_s_timed_region": round(t_wall, 3),
        "clocks": clocks,
    }
    line.update(extra)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows)
    line["headline"] = headline(line)     # last, so a tail of the line keeps it
    print(json.dumps(line), flush=True)


def headline(line: dict) -> dict:
    """The figures the metric is quoted on, compactly: norm+quant us at M=1
    and fraction of HBM per M, the decode step, and the GEMM's TFLOP/s and
    fraction of the FP8 peak at the full-path and long-context sizes."""
    h = {"gemm_dual_M8192_tflops": line["roofline"]["achieved"], "gemm_dual_M8192_frac_fp8": line["roofline"]["frac"]}
    if "norm_quant_us_at_M1" in line:
        h["norm_quant_us_at_M1"] = line["norm_quant_us_at_M1"]
    sw = line.get("norm_quant_sweep", {})
    h["norm_quant_graph_frac_hbm"] = {m: v.get("fused_graph_frac_hbm") for m, v in sw.items() if isinstance(v, dict)}
    h["norm_quant_speedup_vs_unfused"] = {m: v.get("speedup_vs_unfused") for m, v in sw.items() if isinstance(v, dict)}
    h["norm_quant_step_frac_hbm_M8192"] = line["roofline_norm_quant"]["frac"]
    if "decode_step_us_at_M1" in line:
        ds1 = line["decode_step_us_at_M1"]
        h["decode_step_us_at_M1"] = ds1.get("overlap")
        if ds1.get("one_launch") is not None:
            h["decode_step_us_at_M1_one_launch"] = ds1["one_launch"]
    gs = line.get("gemm_sweep", {})
    if "1" in gs:
        h["gemm_dual_M1_graph_us"] = gs["1"].get("graph_us")
        h["gemm_dual_M1_graph_frac_hbm"] = gs["1"].get("graph_frac_hbm")
    if "1024" in gs:
        h["gemm_dual_M1024_tflops"] = gs["1024"].get("tflops")
    if "32768_long_context_attn" in gs:
        h["gemm_attn_M32768_tflops"] = gs["32768_long_context_attn"]["tflops"]
        h["gemm_attn_M32768_frac_fp8"] = gs["32768_long_context_attn"]["frac_fp8"]
    sl = line.get("single_latent_norm_quant", {})
    if "1" in sl:
        h["single_latent_us_at_M1"] = sl["1"]["graph_us"]
        h["single_latent_graph_frac_hbm"] = {m: v["graph_frac_hbm"] for m, v in sl.items()
                                             if isinstance(v, dict) and m != "1"}
    ds = line.get("decode_sweep", {})
    h["norm_quant_decode_us"] = {m: [v["row_us"], v["col_us"]] for m, v in ds.items() if isinstance(v, dict)}
    cb = line.get("cpu_baseline")
    if cb:
        h["cpu_oracle_tflops"] = {"cores": cb["cores"], "all": cb["value"], "one_thread": cb["single_thread"]["value"]}
    return h


def graph_sets(bytes_per_set):
    """Distinct input/output sets for a graph that cycles over them: enough
    that more than 160 MiB (more than L2) of other sets pass between two
    visits of one set."""
    return 1 + max(1, -(-160 * 2 ** 20 // bytes_per_set))


def timed_graph_calls(torch, stream, fn_list, flush, reps=20):
    """Replays a CUDA graph of len(fn_list) calls `reps` times, L2 flushed
    before each replay; returns the median per-call time in microseconds."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        for fn in fn_list:       # warm up on the side stream once
            fn()
    stream.wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for fn in fn_list:
            fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps + 2):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3 / len(fn_list))
    return statistics.median(times[2:])


def side_measurements(torch, dsnq, inputs, dev, flush, hbm_gbs, args, fp8_peak):
    stream = torch.cuda.current_stream()
    out = {}
    # -- M=1 decode latency: 100 calls, each on its own cold row of a split-view buffer
    n = max(100, DECODE_GRAPH_CALLS)       # the decode step below takes its cold rows from here too
    dec = inputs.decode_batch(n, seed=1)
    buf = dec.buf.to(dev)
    gq, gkv = dec.gamma_q.to(dev), dec.gamma_kv.to(dev)
    qo = torch.empty(1, KQ, dtype=torch.float8_e4m3fn, device=dev)
    so = torch.empty(1, KQ // 128, dtype=torch.float32, device=dev)
    ko = torch.empty(1, KKV, dtype=torch.bfloat16, device=dev)
    calls = [(lambda r=r: dsnq.fused_dual_rmsnorm_group_quant(
        buf[r:r + 1, :KQ], buf[r:r + 1, KQ:KQ + KKV], gq, gkv, dec.eps, q_out=qo, q_scale=so, kv_out=ko))
        for r in range(n)]
    out["norm_quant_us_at_M1"] = round(timed_graph_calls(torch, stream, calls, flush), 3)
    dsnq.set_launch_overlap(False)
    out["norm_quant_us_at_M1_no_overlap"] = round(timed_graph_calls(torch, stream, calls, flush), 3)
    dsnq.set_launch_overlap(True)
    out["norm_quant_us_at_M1_note"] = ("per call, CUDA graph of 100 calls on 100 distinct cold rows, L2 flushed per "
                                       "replay; _no_overlap: the same with programmatic dependent launch off")
    out["decode_step_us_at_M1"] = decode_step(torch, dsnq, inputs, dev, flush, buf, gq, gkv, dec.eps, qo, so, ko)
    out["gemm_sweep"] = gemm_sweep(torch, dsnq, inputs, dev, flush, hbm_gbs, args, fp8_peak)
    out["decode_sweep"] = decode_sweep(torch, dsnq, inputs, dev, flush, hbm_gbs)

    # -- norm+quant GB/s over M, and the unfused three-kernel sequence at the same M
    sweep = {}
    for M in args.nq_sweep:
        lat = inputs.prefill_batch(M, seed=2) if M == 8192 else inputs.full_path_batch(M, seed=5)
        q, kv = lat.q.to(dev), lat.kv.to(dev)
        gq2, gkv2 = lat.gamma_q.to(dev), lat.gamma_kv.to(dev)
        qf = torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev)
        sc = dsnq.empty_scales(M, KQ // 128, "col", dev)
        ko2 = torch.empty(M, KKV, dtype=torch.bfloat16, device=dev)
        qb = torch.empty(M, KQ, dtype=torch.bfloat16, device=dev)
        qf2 = torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev)
        sc2 = dsnq.empty_scales(M, KQ // 128, "col", dev)

        def fused():
            dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq2, gkv2, lat.eps, scale_layout="col",
                                                q_out=qf, q_scale=sc, kv_out=ko2)

        def unfused():
            dsnq.dual_rmsnorm_bf16(q, kv, gq2, gkv2, lat.eps, q_out=qb, kv_out=ko2)
            dsnq.group_quant_bf16(qb, scale_layout="col", x_out=qf, x_scale=sc)     # attention wq_b input
            dsnq.group_quant_bf16(qb, scale_layout="col", x_out=qf2, x_scale=sc2)   # indexer wq_b input

        f_us = time_events(torch, stream, fused, flush, reps=args.side_reps)
        u_us = time_events(torch, stream, unfused, flush, reps=args.side_reps)
        gbs = (M * NQ_BYTES_PER_ROW + NQ_BYTES_PER_CALL) / (f_us * 1e-6) / 1e9
        sweep[str(M)] = {"fused_us": round(f_us, 3), "fused_gbs": round(gbs, 1),
                         "fused_frac_hbm": round(gbs / hbm_gbs, 4),
                         "unfused_3_kernels_us": round(u_us, 3),
                         "speedup_vs_unfused": round(u_us / f_us, 3)}
        # Back-to-back calls: a CUDA graph cycling over distinct input/output
        # sets, so every call reads from and writes to HBM.
        nsets = graph_sets(M * NQ_BYTES_PER_ROW)
        if nsets * M * NQ_BYTES_PER_ROW <= 2 * 2 ** 30:
            sets = [(q.clone(), kv.clone(), torch.empty_like(qf), dsnq.empty_scales(M, KQ // 128, "col", dev),
                     torch.empty_like(ko2)) for _ in range(nsets)]
            calls = [(lambda t=sets[i % nsets]: dsnq.fused_dual_rmsnorm_group_quant(
                t[0], t[1], gq2, gkv2, lat.eps, scale_layout="col", q_out=t[2], q_scale=t[3], kv_out=t[4]))
                for i in range(max(nsets, NQ_GRAPH_CALLS))]
            g_us = timed_graph_calls(torch, stream, calls, flush, reps=max(args.side_reps, 5))
            g_gbs = (M * NQ_BYTES_PER_ROW + NQ_BYTES_PER_CALL) / (g_us * 1e-6) / 1e9
            sweep[str(M)].update({"fused_graph_us": round(g_us, 3), "fused_graph_gbs": round(g_gbs, 1),
                                  "fused_graph_frac_hbm": round(g_gbs / hbm_gbs, 4), "graph_sets": nsets,
                                  "graph_calls": len(calls)})
            del sets, calls
        del q, kv, qf, sc, ko2, qb, qf2, sc2
    out["norm_quant_sweep"] = sweep
    out["single_latent_norm_quant"] = single_latent(torch, dsnq, inputs, dev, flush, hbm_gbs, args)
    out["norm_quant_sweep_note"] = ("fused_us / unfused: single launches timed with CUDA events, L2 flushed before "
                                    "each (includes launch latency); fused_graph_us: per call in a CUDA graph of "
                                    "graph_calls back-to-back calls cycling over graph_sets distinct input/output sets "
                                    "(a set comes back only after more than 160 MiB of others, more than L2); M=8192 "
                                    "uses the prefill Student-t inputs, column-major scales")
    return out


def single_latent(torch, dsnq, inputs, dev, flush, hbm_gbs, args):
    """The single-latent RMSNorm + per-1x128 quant (the q latent alone,
    [M, 1536] bf16 -> codes + column-major scales): per call in CUDA graphs,
    M=1 over 100 cold rows and the larger M over input/output sets that
    exceed L2.  Bytes per row: 3072 read, 1536 + 48 written."""
    stream = torch.cuda.current_stream()
    per_row, per_call = KQ * 2 + KQ + 4 * (KQ // 128), KQ * 2
    res = {}
    for M in [1] + [m for m in args.nq_sweep if m >= 1024]:
        x = inputs.full_path_batch(max(M, 100), seed=7).q.to(dev)
        gq = inputs.gammas(8)[0].to(dev)
        if M == 1:
            qf = torch.empty(1, KQ, dtype=torch.float8_e4m3fn, device=dev)
            sc = dsnq.empty_scales(1, KQ // 128, "col", dev)
            calls = [(lambda r=r: dsnq.rmsnorm_group_quant(x[r:r + 1], gq, 1e-6, scale_layout="col",
                                                           x_out=qf, x_scale=sc)) for r in range(100)]
        else:
            nsets = graph_sets(M * per_row)
            sets = [(x[:M].clone(), torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev),
                     dsnq.empty_scales(M, KQ // 128, "col", dev)) for _ in range(nsets)]
            calls = [(lambda s=sets[i % nsets]: dsnq.rmsnorm_group_quant(s[0], gq, 1e-6, scale_layout="col",
                                                                         x_out=s[1], x_scale=s[2]))
                     for i in range(max(nsets, NQ_GRAPH_CALLS))]
        us = timed_graph_calls(torch, stream, calls, flush, reps=max(args.side_reps, 5))
        gbs = (M * per_row + per_call) / (us * 1e-6) / 1e9
        res[str(M)] = {"graph_us": round(us, 3), "graph_gbs": round(gbs, 1), "graph_frac_hbm": round(gbs / hbm_gbs, 4)}
        del calls, x
    res["note"] = ("per call in a CUDA graph: M=1 over 100 distinct cold rows, larger M as at least "
                   f"{NQ_GRAPH_CALLS} calls cycling over distinct input/output sets (a set comes back only after more "
                   "than 160 MiB of others); L2 flushed per replay")
    return res


def decode_sweep(torch, dsnq, inputs, dev, flush, hbm_gbs):
    """Norm+quant at the decode batch sizes, on strided split views of one
    [M, 2112] buffer per call, in both scale layouts: us per call in a CUDA
    graph of DECODE_GRAPH_CALLS calls on as many distinct cold batches (L2
    flushed per replay)."""
    stream = torch.cuda.current_stream()
    res = {}
    for M in (1, 2, 8, 32, 64):
        dec = inputs.decode_batch(DECODE_GRAPH_CALLS * M, seed=1)
        buf = dec.buf.to(dev)
        gq, gkv = dec.gamma_q.to(dev), dec.gamma_kv.to(dev)
        qo = torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev)
        ko = torch.empty(M, KKV, dtype=torch.bfloat16, device=dev)
        r = {}
        for lay in ("row", "col"):
            so = dsnq.empty_scales(M, KQ // 128, lay, dev)
            calls = [(lambda i=i: dsnq.fused_dual_rmsnorm_group_quant(
                buf[i * M:(i + 1) * M, :KQ], buf[i * M:(i + 1) * M, KQ:KQ + KKV], gq, gkv, dec.eps, scale_layout=lay,
                q_out=qo, q_scale=so, kv_out=ko)) for i in range(DECODE_GRAPH_CALLS)]
            r[lay + "_us"] = round(timed_graph_calls(torch, stream, calls, flush), 3)
        res[str(M)] = r
    res["note"] = (f"us per call: CUDA graph of {DECODE_GRAPH_CALLS} calls on as many distinct cold batches of split "
                   "views (row stride 2112), "
                   "L2 flushed per replay; row = [M,12] scales, col = [12,M] (transpose_scale)")
    return res


def decode_step(torch, dsnq, inputs, dev, flush, buf, gq, gkv, eps, qo, so, ko):
    """One decode step at M=1 (fused norm+quant, then the dual GEMM on its
    output): a CUDA graph of DECODE_GRAPH_CALLS steps on as many cold rows,
    cycling over 4 copies of the weights (176 MB, more than L2), with launch
    overlap on and off."""
    stream = torch.cuda.current_stream()
    wa, swa = dsnq.quantize_weight_block128(inputs.weight(N_ATTN, KQ, seed=0, salt=1).to(dev))
    wi, swi = dsnq.quantize_weight_block128(inputs.weight(N_IDX, KQ, seed=0, salt=2).to(dev))
    copies = [(wa, swa, wi, swi)] + [(wa.clone(), swa.clone(), wi.clone(), swi.clone()) for _ in range(3)]
    oa = torch.empty(1, N_ATTN, dtype=torch.bfloat16, device=dev)
    oi = torch.empty(1, N_IDX, dtype=torch.bfloat16, device=dev)

    def step(r, c):
        dsnq.fused_dual_rmsnorm_group_quant(buf[r:r + 1, :KQ], buf[r:r + 1, KQ:KQ + KKV], gq, gkv, eps,
                                            q_out=qo, q_scale=so, kv_out=ko)
        dsnq.block_scaled_fp8_gemm_dual(qo, so, c[0], c[1], c[2], c[3], out1=oa, out2=oi)

    n_steps = DECODE_GRAPH_CALLS
    steps = [(lambda r=r: step(r, copies[r % 4])) for r in range(n_steps)]
    res = {}
    for overlap in (True, False):
        dsnq.set_launch_overlap(overlap)
        res["overlap" if overlap else "no_overlap"] = round(timed_graph_calls(torch, stream, steps, flush), 3)
    dsnq.set_launch_overlap(True)

    # bf16 activations without a pre-quantized pair: quantized inside the GEMM
    # (one launch) against the quant kernel followed by the GEMM.
    xa = inputs.activations_bf16(n_steps, KQ, seed=9).to(dev)
    so_col = dsnq.empty_scales(1, KQ // 128, "col", dev)
    in_gemm = [(lambda r=r: dsnq.block_scaled_fp8_gemm_dual_bf16a(xa[r:r + 1], *copies[r % 4], out1=oa, out2=oi))
               for r in range(n_steps)]

    def two_launches(r):
        dsnq.group_quant_bf16(xa[r:r + 1], scale_layout="col", x_out=qo, x_scale=so_col)
        dsnq.block_scaled_fp8_gemm_dual(qo, so_col, *copies[r % 4], out1=oa, out2=oi)

    res["bf16_in_gemm_quant"] = round(timed_graph_calls(torch, stream, in_gemm, flush), 3)
    res["bf16_quant_then_gemm"] = round(timed_graph_calls(torch, stream, [(lambda r=r: two_launches(r))
                                                                          for r in range(n_steps)], flush), 3)
    one = [(lambda r=r: dsnq.fused_norm_quant_gemm_dual(buf[r:r + 1, :KQ], buf[r:r + 1, KQ:KQ + KKV], gq, gkv, eps,
                                                        *copies[r % 4], out1=oa, out2=oi, kv_out=ko))
           for r in range(n_steps)]
    res["one_launch"] = round(timed_graph_calls(torch, stream, one, flush), 3)
    res["note"] = ("us per step: fused norm+quant then the dual GEMM (44 MB of weights from HBM), CUDA graph of "
                   f"{n_steps} steps on {n_steps} cold rows over 4 weight copies; overlap = programmatic dependent launch (default); "
                   "one_launch: the same step with the norm+quant inside the GEMM; "
                   "bf16_*: the dual GEMM on a bf16 row quantized inside the GEMM, or by the quant kernel first")
    return res


def gemm_sweep(torch, dsnq, inputs, dev, flush, hbm_gbs, args, fp8_peak):
    """The dual GEMM alone over the decode and full-path batch sizes, with
    pre-quantized activations: us per launch, TFLOP/s and weight-stream GB/s."""
    stream = torch.cuda.current_stream()
    wa, swa = dsnq.quantize_weight_block128(inputs.weight(N_ATTN, KQ, seed=0, salt=1).to(dev))
    wi, swi = dsnq.quantize_weight_block128(inputs.weight(N_IDX, KQ, seed=0, salt=2).to(dev))
    wbytes = (N_ATTN + N_IDX) * KQ
    res = {}
    copies = []
    for M in args.gemm_sweep:
        a, sa = inputs.random_codes_and_scales(M, KQ, seed=M)
        a, sa = a.to(dev), sa.to(dev).t().contiguous().t()        # column-major scales, as the path writes them
        oa = torch.empty(M, N_ATTN, dtype=torch.bfloat16, device=dev)
        oi = torch.empty(M, N_IDX, dtype=torch.bfloat16, device=dev)
        us = time_events(torch, stream, lambda: dsnq.block_scaled_fp8_gemm_dual(
            a, sa, wa, swa, wi, swi, out1=oa, out2=oi), flush, reps=args.side_reps)
        byt = wbytes + M * (KQ + 4 * KQ // 128) + 2 * M * (N_ATTN + N_IDX)
        res[str(M)] = {"us": round(us, 3), "tflops": round(gemm_flops(M) / (us * 1e-6) / 1e12, 1),
                       "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                       "frac_hbm": round(byt / (us * 1e-6) / 1e9 / hbm_gbs, 4)}
        if M <= 128:
            # Back-to-back calls as in a decode loop: a CUDA graph of
            # DECODE_GRAPH_CALLS calls over 4 copies of the weights (176 MB, more
            # than L2), so each call streams its weights from HBM without the
            # per-launch host and event overhead.
            if not copies:
                copies.extend([(wa, swa, wi, swi)] + [(wa.clone(), swa.clone(), wi.clone(), swi.clone())
                                                      for _ in range(3)])
            calls = [(lambda c=copies[i % 4]: dsnq.block_scaled_fp8_gemm_dual(
                a, sa, c[0], c[1], c[2], c[3], out1=oa, out2=oi)) for i in range(DECODE_GRAPH_CALLS)]
            gus = timed_graph_calls(torch, stream, calls, flush, reps=max(args.side_reps, 5))
            res[str(M)].update({"graph_us": round(gus, 3), "graph_gbs": round(byt / (gus * 1e-6) / 1e9, 1),
                                "graph_frac_hbm": round(byt / (gus * 1e-6) / 1e9 / hbm_gbs, 4)})
    # Long-context stress: q[32768,1536] with all-zero and single-spike groups,
    # normalized and quantized by the fused kernel (column-major scales), then
    # the attention wq_b GEMM (N=24576) on the pair it wrote.
    if args.long_context:
        M = 32768
        lat = inputs.long_context_batch(M, seed=4)
        q8, s8, _ = dsnq.fused_dual_rmsnorm_group_quant(lat.q.to(dev), lat.kv.to(dev), lat.gamma_q.to(dev),
                                                        lat.gamma_kv.to(dev), lat.eps, scale_layout="col")
        oa = torch.empty(M, N_ATTN, dtype=torch.bfloat16, device=dev)
        us = time_events(torch, stream, lambda: dsnq.block_scaled_fp8_gemm(q8, s8, wa, swa, out=oa), flush,
                         reps=max(5, args.side_reps // 2))
        fl = 2.0 * M * N_ATTN * KQ
        res["32768_long_context_attn"] = {"us": round(us, 3), "tflops": round(fl / (us * 1e-6) / 1e12, 1),
                                          "frac_fp8": round(fl / (us * 1e-6) / 1e12 / fp8_peak, 4),
                                          "kernel": "pair_gemm_kernel", "N": N_ATTN}
        del q8, s8, oa
    res["note"] = ("column-major activation scales; us: one launch timed with CUDA events after an L2 flush (includes "
                   f"launch latency); graph_us: per call in a CUDA graph of {DECODE_GRAPH_CALLS} back-to-back calls over 4 weight copies "
                   "(cold in L2); 32768_long_context_attn: the long-context stress rows quantized by the fused kernel, "
                   "then the attention wq_b GEMM alone (N=24576)")
    return res


def time_events(torch, stream, fn, flush, reps=20):
    for _ in range(3):
        flush()
        fn()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts)


def e2e_measurement(torch, dsnq, lat, dev, weights, args, M):
    """The step through the public API with pinned host buffers: q/kv in,
    both projections and kv out, every copy inside the timed region.

    Steps are pipelined the way a serving loop runs them: the inputs of step
    i+1 are copied in and its kernels run while the outputs of step i are
    still being copied out (three streams, two sets of device buffers, events
    between them).  The device->host copy of the 478 MB of bf16 outputs is
    what bounds the step (about 193 GB/s to pinned host memory on this
    machine, whatever the number of concurrent copies)."""
    wa, swa, wi, swi = weights
    q_h = lat.q.pin_memory()
    kv_h = lat.kv.pin_memory()
    oa_h = torch.empty(M, N_ATTN, dtype=torch.bfloat16).pin_memory()
    oi_h = torch.empty(M, N_IDX, dtype=torch.bfloat16).pin_memory()
    kvo_h = torch.empty(M, KKV, dtype=torch.bfloat16).pin_memory()
    gq, gkv = lat.gamma_q.to(dev), lat.gamma_kv.to(dev)
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def buffers():
        return {"q": torch.empty_like(q_h, device=dev), "kv": torch.empty_like(kv_h, device=dev),
                "q8": torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev),
                "s8": dsnq.empty_scales(M, KQ // 128, "col", dev),
                "kvo": torch.empty(M, KKV, dtype=torch.bfloat16, device=dev),
                "oa": torch.empty(M, N_ATTN, dtype=torch.bfloat16, device=dev),
                "oi": torch.empty(M, N_IDX, dtype=torch.bfloat16, device=dev),
                "in_free": torch.cuda.Event(), "out_free": torch.cuda.Event()}
    sets = [buffers(), buffers()]
    for b in sets:
        b["in_free"].record(s_run)
        b["out_free"].record(s_out)

    def step(i):
        b = sets[i % 2]
        s_in.wait_event(b["in_free"])            # step i-2's kernels have read these inputs
        with torch.cuda.stream(s_in):
            b["q"].copy_(q_h, non_blocking=True)
            b["kv"].copy_(kv_h, non_blocking=True)
        loaded = torch.cuda.Event()
        loaded.record(s_in)
        s_run.wait_event(loaded)
        s_run.wait_event(b["out_free"])          # step i-2's outputs have been copied out
        dsnq.fused_dual_rmsnorm_group_quant(b["q"], b["kv"], gq, gkv, lat.eps, scale_layout="col",
                                            q_out=b["q8"], q_scale=b["s8"], kv_out=b["kvo"], stream=s_run)
        b["in_free"].record(s_run)
        dsnq.block_scaled_fp8_gemm_dual(b["q8"], b["s8"], wa, swa, wi, swi, out1=b["oa"], out2=b["oi"],
                                        stream=s_run)
        done = torch.cuda.Event()
        done.record(s_run)
        s_out.wait_event(done)
        with torch.cuda.stream(s_out):
            oa_h.copy_(b["oa"], non_blocking=True)
            oi_h.copy_(b["oi"], non_blocking=True)
            kvo_h.copy_(b["kvo"], non_blocking=True)
        b["out_free"].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    reps = max(4, min(args.steps, 20))
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(reps):
        step(i)
    s_in.wait_stream(s_out)
    z.record(s_in)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / reps
    # Every step copies out the same products: the host buffers must hold
    # exactly those of a plain call (a race between the streams would not).
    q8, s8, kvo = dsnq.fused_dual_rmsnorm_group_quant(q_h.to(dev), kv_h.to(dev), gq, gkv, lat.eps, scale_layout="col")
    ra, ri = dsnq.block_scaled_fp8_gemm_dual(q8, s8, wa, swa, wi, swi)
    torch.cuda.synchronize(dev)
    for host, want in ((oa_h, ra), (oi_h, ri), (kvo_h, kvo)):
        if not torch.equal(host.view(torch.int16), want.view(torch.int16).cpu()):
            raise RuntimeError("e2e: the outputs copied out by the pipelined steps differ from a plain call")
    h2d = q_h.numel() * 2 + kv_h.numel() * 2
    d2h = (oa_h.numel() + oi_h.numel() + kvo_h.numel()) * 2
    return {"value": round(gemm_flops(M) / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "public API on three streams (copy in, kernels, copy out), consecutive steps overlapped"}


# ----------------------------------------------------------------- CPU oracle

_SAMPLE_CACHE = {}


def _sample_inputs(rows, cols_per_consumer, seed, M):
    """Synthetic inputs of one oracle sample (generated once; not timed)."""
    key = (rows, cols_per_consumer, seed, M)
    if key not in _SAMPLE_CACHE:
        import numpy as np
        import oracle
        from gemm_dsnq_dual_gb300 import inputs
        lat = inputs.full_path_batch(M, seed=seed)
        if rows > M:
            raise ValueError(f"a sample of {rows} rows does not fit the M={M} workload")
        pick = np.random.default_rng(0).choice(M, rows, replace=False)
        b = [inputs.bits(t) for t in (lat.q[pick], lat.kv[pick], lat.gamma_q, lat.gamma_kv)]
        weights = []
        for N, salt in ((N_ATTN, 1), (N_IDX, 2)):
            n = N if cols_per_consumer is None else min(N, cols_per_consumer)
            w = inputs.weight(N, KQ, seed=0, salt=salt)[:n].numpy()
            weights.append(oracle.quantize_weight_block128(w))   # load-time weight prep
        _SAMPLE_CACHE[key] = (b, lat.eps, weights)
    return _SAMPLE_CACHE[key]


def oracle_full_path_sample(rows: int, cols_per_consumer, seed=3, M=8192):
    """One bounded sample of the full-path workload through the fp64 oracle:
    norm+quant of `rows` token rows, then the block-scaled GEMM of those rows
    against `cols_per_consumer` (None = all) output features of each wq_b.
    Returns (seconds, flops)."""
    import oracle
    b, eps, weights = _sample_inputs(rows, cols_per_consumer, seed, M)
    t0 = time.perf_counter()
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(*b, eps)
    flops = 0.0
    for wc, ws in weights:
        oracle.output_bf16_bits(oracle.block_scaled_gemm(codes, scale, wc, ws))
        flops += 2.0 * rows * wc.shape[0] * KQ
    return time.perf_counter() - t0, flops


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
               "NUMEXPR_NUM_THREADS")


def oracle_child(threads: int, rows: int):
    """Runs in a child process with a one-thread BLAS pool: the oracle on
    `rows` rows of the M=8192 full path, spread over `threads` worker threads
    (numpy releases the GIL in its array operations): the norm+quant by row
    ranges, the GEMM by 128-row blocks of the weights.  Prints one JSON line."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import oracle
    b, eps, weights = _sample_inputs(rows, None, 3, 8192)
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda c: oracle.fused_dual_rmsnorm_group_quant(b[0][c], b[1][c], b[2], b[3], eps)[:2],
                            np.array_split(np.arange(rows), threads)))
        codes = np.concatenate([p[0] for p in parts])
        scale = np.concatenate([p[1] for p in parts])
        flops = 0.0
        for wc, ws in weights:
            nb = ws.shape[0]
            spans = [(int(c[0]), int(c[-1]) + 1) for c in np.array_split(np.arange(nb), min(threads, nb)) if len(c)]
            outs = list(ex.map(lambda sp: oracle.block_scaled_gemm(codes, scale, wc[sp[0] * 128:sp[1] * 128],
                                                                   ws[sp[0]:sp[1]]), spans))
            oracle.output_bf16_bits(np.concatenate(outs, axis=1))
            flops += 2.0 * rows * wc.shape[0] * KQ
    secs = time.perf_counter() - t0
    print(json.dumps({"secs": secs, "flops": flops, "threads": threads}), flush=True)


def oracle_timed(threads: int, rows: int):
    """The oracle timed in a fresh process with `threads` worker threads and a
    one-thread BLAS pool (a child process, so the pool size is set before
    numpy loads and nothing is forked from a process that used the GPU)."""
    env = dict(os.environ)
    for k in _THREAD_ENV:
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(threads), "--cpu-rows",
                        str(rows)], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(rows: int):
    """The fp64 oracle on the host: `rows` random rows of the M=8192 full
    path (norm+quant, then the GEMM against all 24576+4096 features), once
    on one thread and once on all the host's cores."""
    n = host_cores()
    one = oracle_timed(1, rows)
    alln = oracle_timed(n, rows)
    sample = (f"{rows} random rows of the M=8192 full path: fp64 norm+quant, then the dequantize-then-fp64 GEMM "
              f"against all 24576+4096 features")
    return {"value": round(alln["flops"] / alln["secs"] / 1e12, 6), "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "sample": f"{sample} ({alln['secs']:.1f} s on {n} threads)",
            "single_thread": {"value": round(one["flops"] / one["secs"] / 1e12, 6), "cores": 1,
                              "secs": round(one["secs"], 2)}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    rows, cols = 32, 256
    for _ in range(args.warmup):
        oracle_full_path_sample(rows, cols)
    tot_s, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        s, f = oracle_full_path_sample(rows, cols)
        tot_s += s
        tot_f += f
    value = tot_f / tot_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(args.M, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"per step: {rows} random rows x {cols} features of each wq_b, "
                                   f"fp64 norm+quant + dequantize-then-fp64 GEMM"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- plumbing

def rank_seed(rank: int) -> int:
    """Seed of the token batch a rank processes: ranks shard the work by
    taking independent batches (weak scaling, no data exchange)."""
    return 3 + rank


def whole_job_value(world: int, flops_per_rank_step: float, step_ms_max: float) -> float:
    """TFLOP/s of the whole job: the work of all ranks over the slowest
    rank's step time."""
    return world * flops_per_rank_step / (step_ms_max * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world, dev):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_kernel_only(args):
    """A few launches of one kernel on the configured workload, for profilers
    (ncu): `--kernel-only gemm` runs the dual GEMM, `norm_quant` the fused
    norm+quant, `single_latent` the single-latent norm+quant of q,
    `unfused` the unfused baseline's three launches (norm to bf16, then the
    quant of q twice), `fused_step` the one-launch norm+quant+GEMM (a few
    decode rows), `bf16a` the dual GEMM on the bf16 q rows (quantized inside
    the GEMM for a few rows); no timing, no JSON line.  Every mode first runs one fused
    norm+quant to make its inputs."""
    import torch
    import gemm_dsnq_dual_gb300 as dsnq
    from gemm_dsnq_dual_gb300 import inputs
    dev = torch.device("cuda", 0)
    M = args.M
    lat = inputs.full_path_batch(M, seed=3)
    q, kv = lat.q.to(dev), lat.kv.to(dev)
    gq, gkv = lat.gamma_q.to(dev), lat.gamma_kv.to(dev)
    q8, s8, _ = dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="col")
    if args.kernel_only in ("gemm", "fused_step", "bf16a"):
        wa, swa = dsnq.quantize_weight_block128(inputs.weight(N_ATTN, KQ, seed=0, salt=1).to(dev))
        wi, swi = dsnq.quantize_weight_block128(inputs.weight(N_IDX, KQ, seed=0, salt=2).to(dev))
    if args.kernel_only == "gemm":
        fn = lambda: dsnq.block_scaled_fp8_gemm_dual(q8, s8, wa, swa, wi, swi)
    elif args.kernel_only == "fused_step":
        # The decode step as one launch (norm+quant inside the GEMM's prologue).
        fn = lambda: dsnq.fused_norm_quant_gemm_dual(q, kv, gq, gkv, lat.eps, wa, swa, wi, swi)
    elif args.kernel_only == "bf16a":
        fn = lambda: dsnq.block_scaled_fp8_gemm_dual_bf16a(q, wa, swa, wi, swi)
    elif args.kernel_only == "single_latent":
        fn = lambda: dsnq.rmsnorm_group_quant(q, gq, lat.eps, scale_layout="col", x_out=q8, x_scale=s8)
    elif args.kernel_only == "unfused":
        qb = torch.empty(M, KQ, dtype=torch.bfloat16, device=dev)
        kb = torch.empty(M, KKV, dtype=torch.bfloat16, device=dev)
        q8b, s8b = torch.empty_like(q8), dsnq.empty_scales(M, KQ // 128, "col", dev)

        def fn():
            dsnq.dual_rmsnorm_bf16(q, kv, gq, gkv, lat.eps, q_out=qb, kv_out=kb)
            dsnq.group_quant_bf16(qb, scale_layout="col", x_out=q8, x_scale=s8)
            dsnq.group_quant_bf16(qb, scale_layout="col", x_out=q8b, x_scale=s8b)
    else:
        fn = lambda: dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="col",
                                                         q_out=q8, q_scale=s8)
    for _ in range(args.launches):
        fn()
    torch.cuda.synchronize()
    print(f"kernel-only {args.kernel_only} M={M}: {args.launches} launches ok")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--nq-sweep", type=int, nargs="*", default=[1024, 8192, 32768])
    ap.add_argument("--side-reps", type=int, default=20)
    ap.add_argument("--gemm-sweep", type=int, nargs="*", default=[1, 8, 64, 128, 1024])
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--no-long-context", dest="long_context", action="store_false",
                    help="skip the M=32768 long-context GEMM of the side measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-only", choices=["gemm", "norm_quant", "single_latent", "unfused", "fused_step", "bf16a"],
                    default=None,
                    help="profiling aid: launch one kernel --launches times and exit")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--oracle-child", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(args.oracle_child, args.cpu_rows)
        return
    if args.kernel_only:
        run_kernel_only(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
