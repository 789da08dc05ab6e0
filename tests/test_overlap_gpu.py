"""Launch overlap (programmatic dependent launch) changes no result.

Every kernel of the library may be scheduled while the previous kernel of its
stream runs, and waits in hardware for that kernel's writes before touching
an argument buffer.  These tests enqueue dependent chains with no host
synchronization in between: each norm+quant overwrites the activation
buffers that the previous GEMM read (write-after-read), each GEMM reads what
the norm+quant just wrote (read-after-write), and the weights are quantized by
the kernel right before the first GEMM.  The outputs with overlap on must be
bit-identical to those with plain stream ordering, and one step is checked
against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import GEMM_REL_FRO, assert_bf16_close, assert_codes_close, assert_scales_close, bf16_value, rel_fro

pytestmark = pytest.mark.gpu

KQ, KKV, N_ATTN, N_IDX = 1536, 512, 24576, 4096


def run_chain(M: int, steps: int, overlap: bool):
    """`steps` decode-style steps sharing one set of activation buffers."""
    dsnq.set_launch_overlap(overlap)
    try:
        dev = torch.device("cuda")
        batches = [inputs.full_path_batch(M, seed=100 + i) for i in range(steps)]
        qs = [b.q.to(dev) for b in batches]
        kvs = [b.kv.to(dev) for b in batches]
        gq, gkv, eps = batches[0].gamma_q.to(dev), batches[0].gamma_kv.to(dev), batches[0].eps
        w_attn = inputs.weight(N_ATTN, KQ, seed=0, salt=1).to(dev)
        w_idx = inputs.weight(N_IDX, KQ, seed=0, salt=2).to(dev)
        torch.cuda.synchronize()
        # Weight quantization immediately followed by the GEMMs that read it.
        wa, swa = dsnq.quantize_weight_block128(w_attn)
        wi, swi = dsnq.quantize_weight_block128(w_idx)
        q8 = torch.empty(M, KQ, dtype=torch.float8_e4m3fn, device=dev)
        s8 = dsnq.empty_scales(M, KQ // 128, "col", device=dev)
        outs = []
        for i in range(steps):
            kv_out = torch.empty(M, KKV, dtype=torch.bfloat16, device=dev)
            dsnq.fused_dual_rmsnorm_group_quant(qs[i], kvs[i], gq, gkv, eps, scale_layout="col",
                                                q_out=q8, q_scale=s8, kv_out=kv_out)
            oa, oi = dsnq.block_scaled_fp8_gemm_dual(q8, s8, wa, swa, wi, swi)
            outs.append((kv_out, oa, oi))
        torch.cuda.synchronize()
        last = (q8.view(torch.uint8).clone(), s8.clone())
        return batches, outs, last, (wa, swa, wi, swi)
    finally:
        dsnq.set_launch_overlap(True)


def bits(t: torch.Tensor) -> torch.Tensor:
    """The raw storage words of a tensor (exact comparison for any dtype)."""
    return t.contiguous().view({1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()])


@pytest.mark.parametrize("M", [1, 200, 2048])
def test_overlap_is_bit_identical(M):
    steps = 6
    _, on, last_on, w_on = run_chain(M, steps, True)
    _, off, last_off, w_off = run_chain(M, steps, False)
    for a, b in zip(w_on, w_off):
        assert torch.equal(bits(a), bits(b))
    assert torch.equal(last_on[0], last_off[0]) and torch.equal(bits(last_on[1]), bits(last_off[1]))
    for i, (x, y) in enumerate(zip(on, off)):
        for t_on, t_off in zip(x, y):
            assert torch.equal(bits(t_on), bits(t_off)), f"step {i} differs with overlap on"


def test_overlap_chain_matches_oracle():
    """The last step of an overlapped chain against the oracle (sampled rows)."""
    M, steps = 300, 4
    batches, outs, (q8, s8), (wa, swa, wi, swi) = run_chain(M, steps, True)
    b, g = batches[-1], batches[0]     # every step is normalized with the first batch's gamma
    codes, scale, kv_bits = oracle.fused_dual_rmsnorm_group_quant(
        inputs.bits(b.q), inputs.bits(b.kv), inputs.bits(g.gamma_q), inputs.bits(g.gamma_kv), g.eps)
    got_codes = q8.cpu().numpy()
    got_scale = s8.cpu().numpy()
    assert_codes_close(got_codes, codes)
    assert_scales_close(got_scale, scale)
    kv_out, oa, oi = outs[-1]
    assert_bf16_close(kv_out.view(torch.int16).cpu().numpy().view(np.uint16), kv_bits)
    rows = np.arange(0, M, 37)
    for out, w, ws in ((oa, wa, swa), (oi, wi, swi)):
        ref = oracle.block_scaled_gemm(got_codes, got_scale, w.view(torch.uint8).cpu().numpy(), ws.cpu().numpy(),
                                       rows=rows)
        got = bf16_value(out[torch.as_tensor(rows, device=out.device)])
        assert rel_fro(got, ref) <= GEMM_REL_FRO
