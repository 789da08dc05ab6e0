"""The bf16-activation dual GEMM with the library's own device scratch for
the quantized pair (no workspace argument, nothing allocated): same results
as the call with a caller workspace, bit for bit, on both routes (quantized
inside the GEMM for a few rows; quant kernel, then the GEMM, above), and
parity with the oracle."""

import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import GEMM_REL_FRO, bf16_value, rel_fro

pytestmark = pytest.mark.gpu


def weights(K):
    out = []
    for N, seed in ((512, 91), (256, 92)):
        wc, ws = oracle.quantize_weight_block128(inputs.weight(N, K, seed=seed).numpy())
        out += [wc, ws]
    return out


@pytest.mark.parametrize("M,K", [(1, 1536), (7, 1536), (300, 1536), (2048, 2048)])
def test_static_scratch_equals_workspace(M, K):
    a = inputs.activations_bf16(M, K, seed=93 + M).cuda()
    w1, s1, w2, s2 = weights(K)
    W = [torch.from_numpy(x).cuda() for x in (w1, s1, w2, s2)]
    o1 = torch.empty(M, 512, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty(M, 256, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    dsnq.block_scaled_fp8_gemm_dual_bf16a_static(a, *W, out1=o1, out2=o2)   # may load the device code
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before       # no tensor allocated for the call
    # A second call: neither torch's allocator nor the device as a whole
    # (a cudaMalloc inside the library would show there) loses memory.
    free_before = torch.cuda.mem_get_info()[0]
    dsnq.block_scaled_fp8_gemm_dual_bf16a_static(a, *W, out1=o1, out2=o2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.cuda.memory_allocated() == before
    r1, r2 = dsnq.block_scaled_fp8_gemm_dual_bf16a(a, *W)
    assert torch.equal(o1, r1) and torch.equal(o2, r2)
    if M == 300:
        codes, scale = oracle.group_quant_bf16(inputs.bits(a.cpu()))
        ref = oracle.block_scaled_gemm(codes, scale, w1, s1)
        assert rel_fro(bf16_value(o1), ref) <= GEMM_REL_FRO


_FIRST_CALL_IN_CAPTURE = textwrap.dedent("""
    import torch
    import gemm_dsnq_dual_gb300 as dsnq
    from gemm_dsnq_dual_gb300 import inputs
    M, K = 300, 1536
    a = inputs.activations_bf16(M, K, seed=95).cuda()
    W = []
    for N, seed in ((512, 91), (256, 92)):
        W += list(dsnq.quantize_weight_block128(inputs.weight(N, K, seed=seed).cuda()))
    o1 = torch.empty(M, 512, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty(M, 256, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):          # the process's first call of the static entry
        dsnq.block_scaled_fp8_gemm_dual_bf16a_static(a, *W, out1=o1, out2=o2)
    g.replay()
    torch.cuda.synchronize()
    r1, r2 = dsnq.block_scaled_fp8_gemm_dual_bf16a(a, *W)
    assert torch.equal(o1, r1) and torch.equal(o2, r2)
    print("first static call inside capture: ok")
""")


def test_first_static_call_inside_graph_capture():
    """A fresh process whose first call of the static entry (the one that
    looks the array's address up) is made while a CUDA graph is captured:
    the capture succeeds and its replay equals the workspace call."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "ok" in r.stdout
