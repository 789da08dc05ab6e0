"""The dual GEMM on bf16 activations quantized per 1x128 on the fly (the
linear path without a pre-quantized input, sglang PR #27289,
aiter_w8a8_block_fp8_linear): parity with the oracle's group quant of the
same bf16 rows followed by its fp64 block-scaled product.  At decode sizes
the GEMM quantizes inside the kernel; larger batches run the quant kernel
into a workspace and then the GEMM.  Both routes take the same code and
scale decisions, so their outputs are bit-identical."""

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import GEMM_REL_FRO, bf16_value, rel_fro

pytestmark = pytest.mark.gpu


def quantized_weight(N, K, seed, salt=0):
    return oracle.quantize_weight_block128(inputs.weight(N, K, seed=seed, salt=salt).numpy())


def dev(*arrays):
    return [torch.from_numpy(x).cuda() for x in arrays]


def check_against_oracle(out, a_bits, wc, ws, rows=None):
    codes, scale = oracle.group_quant_bf16(a_bits)
    ref = oracle.block_scaled_gemm(codes, scale, wc, ws, rows=rows)
    got = bf16_value(out if rows is None else out[torch.as_tensor(rows, device=out.device)])
    err = rel_fro(got, ref)
    assert err <= GEMM_REL_FRO, err


SHAPES = [
    # M, K, N1, N2
    (1, 1536, 512, 256),    # quantized inside the GEMM ...
    (6, 1536, 256, 128),
    (5, 384, 256, 0),       # odd number of K blocks
    (16, 128, 128, 128),    # one K block, 16 rows (two launches: more than 8 rows)
    (8, 128, 128, 128),     # one K block, 8 rows: every resident row live, the MMA's rows 8..15 in the spare block
    (8, 1280, 256, 128),    # 8 rows x 5 slots = 40 units: the in-GEMM bound
    (2, 2048, 256, 0),      # largest K quantized in the GEMM
    (7, 1536, 512, 256),    # ... and the quant kernel, then the GEMM
    (17, 1536, 512, 256),
    (64, 1664, 384, 256),   # odd number of K blocks
    (65, 1536, 512, 256),   # 128x128 tiles
    (300, 1536, 256, 512),  # CTA pairs
]


@pytest.mark.parametrize("M,K,N1,N2", SHAPES)
def test_bf16a_matches_oracle(M, K, N1, N2):
    a = inputs.activations_bf16(M, K, seed=M + K, zero_rows=(M // 2,) if M > 2 else ())
    w1, s1 = quantized_weight(N1, K, seed=N1 + K)
    w2, s2 = quantized_weight(max(N2, 16), K, seed=N2 + K + 1)
    W1, S1, W2, S2 = dev(w1, s1, w2[:N2], s2[: (N2 + 127) // 128])
    o1, o2 = dsnq.block_scaled_fp8_gemm_dual_bf16a(a.cuda(), W1, S1, W2, S2)
    torch.cuda.synchronize()
    bits = inputs.bits(a)
    check_against_oracle(o1, bits, w1, s1)
    if N2:
        check_against_oracle(o2, bits, w2[:N2], s2[: (N2 + 127) // 128])
    if M > 2:
        assert not o1[M // 2].any()          # an all-zero row: scale 0, codes 0, output 0


@pytest.mark.parametrize("M", [1, 2, 5, 6])
def test_in_gemm_quant_equals_quant_kernel_then_gemm(M):
    K = 1536
    a = inputs.activations_bf16(M, K, seed=50 + M).cuda()
    w1, s1 = quantized_weight(1024, K, seed=51)
    w2, s2 = quantized_weight(256, K, seed=52)
    W1, S1, W2, S2 = dev(w1, s1, w2, s2)
    assert dsnq.fused_quant_fits(M, K)
    f1, f2 = dsnq.block_scaled_fp8_gemm_dual_bf16a(a, W1, S1, W2, S2)
    codes, scale = dsnq.group_quant_bf16(a, scale_layout="col")
    t1, t2 = dsnq.block_scaled_fp8_gemm_dual(codes, scale, W1, S1, W2, S2)
    assert torch.equal(f1, t1) and torch.equal(f2, t2)


def test_bf16a_decode_full_width():
    """M=1 against both wq_b at full width (44 MB of weights)."""
    K = inputs.KQ
    a = inputs.activations_bf16(1, K, seed=60)
    wa, swa = quantized_weight(inputs.N_ATTN, K, seed=0, salt=1)
    wi, swi = quantized_weight(inputs.N_IDX, K, seed=0, salt=2)
    oa, oi = dsnq.block_scaled_fp8_gemm_dual_bf16a(a.cuda(), *dev(wa, swa, wi, swi))
    torch.cuda.synchronize()
    bits = inputs.bits(a)
    check_against_oracle(oa, bits, wa, swa)
    check_against_oracle(oi, bits, wi, swi)
