"""Parity of the tcgen05 block-scaled FP8 GEMM with the fp64 dequantized
product of the oracle, through the C ABI: small and ragged shapes in both
orientations (decode swap-AB and large M), both activation-scale layouts, the
dual-consumer launch, the full path at the workload sizes (fused norm+quant
feeding attention wq_b N=24576 and indexer wq_b N=4096 over K=1536, checked on
sampled rows), the long-context stress, and the bounded-wait timeout."""

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import GEMM_REL_FRO, bf16_value, rel_fro

pytestmark = pytest.mark.gpu


def scales_in_layout(sa: torch.Tensor, layout, pad=0) -> torch.Tensor:
    """The logical [M, G] scales copied into a device buffer of the layout."""
    M, G = sa.shape
    if layout == dsnq.ROW_MAJOR:
        buf = torch.zeros(M, G + pad, dtype=torch.float32, device="cuda")
        buf[:, :G] = sa.cuda()
        return buf[:, :G]
    buf = torch.zeros(G, M + pad, dtype=torch.float32, device="cuda")
    buf[:, :M] = sa.cuda().t()
    return buf[:, :M].t()


def quantized_weight(N, K, seed, salt=0):
    w = inputs.weight(N, K, seed=seed, salt=salt).numpy()
    return oracle.quantize_weight_block128(w)


def check_gemm(got_bf16: torch.Tensor, a_codes, a_scale, w_codes, w_scale, rows=None):
    ref = oracle.block_scaled_gemm(a_codes, a_scale, w_codes, w_scale, rows=rows)
    got = bf16_value(got_bf16 if rows is None else got_bf16[torch.as_tensor(rows, device=got_bf16.device)])
    err = rel_fro(got, ref)
    assert err <= GEMM_REL_FRO, f"rel-Frobenius {err:.3e}"
    # elementwise: bf16 rounding plus a small multiple of the magnitude of the terms
    A = np.abs(oracle.dequantize_activation(a_codes if rows is None else a_codes[rows],
                                            a_scale if rows is None else a_scale[rows]))
    mag = A @ np.abs(oracle.dequantize_weight(w_codes, w_scale)).T
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -9 * mag + 1e-30
    assert np.all(np.abs(got - ref) <= bound), f"max excess {np.max(np.abs(got - ref) - bound):.3e}"
    return err


# From 256 rows on the GEMM runs in 2 x 2 clusters: odd tile counts along
# either side (300, 520 rows; 128, 272, 656 features) leave padding tiles.
SHAPES = [(1, 128, 128), (3, 256, 256), (16, 512, 1536), (17, 272, 512), (40, 4096, 1536),
          (64, 384, 1536), (65, 256, 384), (128, 512, 1536), (200, 1024, 1536), (300, 272, 768),
          (256, 128, 1536), (520, 656, 256), (1000, 400, 1280)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_gemm_shapes(M, N, K, layout):
    a, sa = inputs.random_codes_and_scales(M, K, seed=M + N)
    wc, ws = quantized_weight(N, K, seed=N + K)
    out = dsnq.block_scaled_fp8_gemm(a.cuda(), scales_in_layout(sa, layout, pad=2),
                                     torch.from_numpy(wc).cuda(), torch.from_numpy(ws).cuda())
    torch.cuda.synchronize()
    check_gemm(out, a.numpy(), sa.numpy(), wc, ws)


# Long K: each kernel variant at the largest K it serves, and the variant
# that takes over beyond it (the plan is checked too, so every variant of
# dsnq_gemm_plan is reached here).
LONG_K = [(1, 256, 8192, 1), (20, 256, 8192, 2), (40, 384, 8192, 3), (100, 256, 4096, 4),
          (100, 256, 4224, 5), (200, 256, 8192, 5), (300, 256, 4096, 6), (300, 256, 4224, 5),
          (520, 384, 8192, 5)]


@pytest.mark.parametrize("M,N,K,variant", LONG_K)
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_gemm_long_k_every_variant(M, N, K, variant, layout):
    assert dsnq.gemm_plan(M, K)[0] == variant
    a, sa = inputs.random_codes_and_scales(M, K, seed=M + K)
    wc, ws = quantized_weight(N, K, seed=N + K + 1)
    out = dsnq.block_scaled_fp8_gemm(a.cuda(), scales_in_layout(sa, layout, pad=1),
                                     torch.from_numpy(wc).cuda(), torch.from_numpy(ws).cuda())
    torch.cuda.synchronize()
    check_gemm(out, a.numpy(), sa.numpy(), wc, ws)


def test_output_guard_and_padded_strides():
    M, N, K = 70, 384, 512
    a, sa = inputs.random_codes_and_scales(M, K, seed=1)
    wc, ws = quantized_weight(N, K, seed=2)
    abuf = torch.zeros(M, K + 32, dtype=torch.uint8, device="cuda")
    abuf[:, :K] = a.cuda()
    wbuf = torch.zeros(N, K + 16, dtype=torch.uint8, device="cuda")
    wbuf[:, :K] = torch.from_numpy(wc).cuda()
    obuf = torch.full((M + 2, N + 24), -7.0, dtype=torch.bfloat16, device="cuda")
    out = obuf[1:M + 1, 8:8 + N]
    dsnq.block_scaled_fp8_gemm(abuf[:, :K], scales_in_layout(sa, dsnq.COL_MAJOR, pad=5), wbuf[:, :K],
                               torch.from_numpy(ws).cuda(), out=out)
    torch.cuda.synchronize()
    check_gemm(out, a.numpy(), sa.numpy(), wc, ws)
    mask = torch.ones_like(obuf, dtype=torch.bool)
    mask[1:M + 1, 8:8 + N] = False
    assert torch.all(obuf[mask] == -7.0)


@pytest.mark.parametrize("M", [5, 300])
def test_row_and_column_major_scales_give_identical_output(M):
    # The silent bug class of vLLM PR #56433: a GEMM reading row-major scales
    # as column-major is only wrong for M > 1.  Both layouts must agree bit for bit.
    N, K = 512, 1536
    a, sa = inputs.random_codes_and_scales(M, K, seed=11)
    wc, ws = quantized_weight(N, K, seed=12)
    w, s = torch.from_numpy(wc).cuda(), torch.from_numpy(ws).cuda()
    o1 = dsnq.block_scaled_fp8_gemm(a.cuda(), scales_in_layout(sa, dsnq.ROW_MAJOR), w, s)
    o2 = dsnq.block_scaled_fp8_gemm(a.cuda(), scales_in_layout(sa, dsnq.COL_MAJOR), w, s)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("M", [8, 256])
def test_dual_launch_equals_two_single_launches(M):
    K = 1536
    a, sa = inputs.random_codes_and_scales(M, K, seed=21)
    w1, s1 = quantized_weight(1024, K, seed=22)
    w2, s2 = quantized_weight(384, K, seed=23)
    A, S = a.cuda(), scales_in_layout(sa, dsnq.COL_MAJOR)
    d1, d2 = dsnq.block_scaled_fp8_gemm_dual(A, S, torch.from_numpy(w1).cuda(), torch.from_numpy(s1).cuda(),
                                             torch.from_numpy(w2).cuda(), torch.from_numpy(s2).cuda())
    o1 = dsnq.block_scaled_fp8_gemm(A, S, torch.from_numpy(w1).cuda(), torch.from_numpy(s1).cuda())
    o2 = dsnq.block_scaled_fp8_gemm(A, S, torch.from_numpy(w2).cuda(), torch.from_numpy(s2).cuda())
    assert torch.equal(d1, o1) and torch.equal(d2, o2)
    check_gemm(d2, a.numpy(), sa.numpy(), w2, s2)


@pytest.fixture(scope="module")
def wq_b_weights():
    """Attention wq_b [24576,1536] and indexer wq_b [4096,1536], N(0,0.02),
    quantized per 128x128 block by the oracle."""
    wa = quantized_weight(inputs.N_ATTN, inputs.KQ, seed=0, salt=1)
    wi = quantized_weight(inputs.N_IDX, inputs.KQ, seed=0, salt=2)
    return wa, wi


@pytest.mark.parametrize("M", [1, 2, 8, 32, 64])
def test_decode_gemm_full_width(M, wq_b_weights):
    (wa, sa_w), _ = wq_b_weights
    a, sa = inputs.random_codes_and_scales(M, inputs.KQ, seed=40 + M)
    out = dsnq.block_scaled_fp8_gemm(a.cuda(), scales_in_layout(sa, dsnq.ROW_MAJOR),
                                     torch.from_numpy(wa).cuda(), torch.from_numpy(sa_w).cuda())
    torch.cuda.synchronize()
    check_gemm(out, a.numpy(), sa.numpy(), wa, sa_w)


@pytest.mark.parametrize("M", [128, 1024, 8192])
def test_full_path_sampled_rows(M, wq_b_weights):
    """Fused norm+quant -> dual GEMM on the GPU, oracle on sampled rows."""
    (wa, swa), (wi, swi) = wq_b_weights
    lat = inputs.full_path_batch(M, seed=3)
    q_fp8, q_scale, _ = dsnq.fused_dual_rmsnorm_group_quant(
        lat.q.cuda(), lat.kv.cuda(), lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps, scale_layout="col")
    oa, oi = dsnq.block_scaled_fp8_gemm_dual(q_fp8, q_scale, torch.from_numpy(wa).cuda(),
                                             torch.from_numpy(swa).cuda(), torch.from_numpy(wi).cuda(),
                                             torch.from_numpy(swi).cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, min(M, 48), replace=False)]))
    b = [inputs.bits(t) for t in (lat.q[rows], lat.kv[rows], lat.gamma_q, lat.gamma_kv)]
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(*b, lat.eps)
    full_codes = np.zeros((M, inputs.KQ), np.uint8)
    full_scale = np.zeros((M, inputs.KQ // 128), np.float32)
    full_codes[rows], full_scale[rows] = codes, scale
    check_gemm(oa, full_codes, full_scale, wa, swa, rows=rows)
    check_gemm(oi, full_codes, full_scale, wi, swi, rows=rows)


def test_long_context_attention_gemm_sampled(wq_b_weights):
    (wa, swa), _ = wq_b_weights
    M = 32768
    lat = inputs.long_context_batch(M, seed=4)
    q_fp8, q_scale, _ = dsnq.fused_dual_rmsnorm_group_quant(
        lat.q.cuda(), lat.kv.cuda(), lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps, scale_layout="col")
    out = dsnq.block_scaled_fp8_gemm(q_fp8, q_scale, torch.from_numpy(wa).cuda(), torch.from_numpy(swa).cuda())
    torch.cuda.synchronize()
    rows = np.array(sorted({0, 97, 89, 89 * 97, M - 1} | set(np.random.default_rng(1).choice(M, 24).tolist())))
    b = [inputs.bits(t) for t in (lat.q[rows], lat.kv[rows], lat.gamma_q, lat.gamma_kv)]
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(*b, lat.eps)
    full_codes = np.zeros((M, inputs.KQ), np.uint8)
    full_scale = np.zeros((M, inputs.KQ // 128), np.float32)
    full_codes[rows], full_scale[rows] = codes, scale
    check_gemm(out, full_codes, full_scale, wa, swa, rows=rows)
    assert torch.all(out[0] == 0) and torch.all(out[M - 1] == 0)     # all-zero rows


def test_gemm_zero_rows():
    out = dsnq.block_scaled_fp8_gemm(torch.empty(0, 1536, dtype=torch.uint8, device="cuda"),
                                     torch.empty(0, 12, device="cuda"),
                                     torch.zeros(256, 1536, dtype=torch.uint8, device="cuda"),
                                     torch.ones(2, 12, device="cuda"))
    assert out.shape == (0, 256)


@pytest.mark.parametrize("M", [4, 200, 512])
def test_bounded_wait_times_out_and_context_survives(M):
    """The producer skips its first load on purpose; the consumer's bounded
    wait runs out, the kernel records a timeout and returns, and the next
    launch on the same context is correct."""
    N, K = 256, 1536
    a, sa = inputs.random_codes_and_scales(M, K, seed=5)
    wc, ws = quantized_weight(N, K, seed=6)
    args = (a.cuda(), scales_in_layout(sa, dsnq.ROW_MAJOR), torch.from_numpy(wc).cuda(),
            torch.from_numpy(ws).cuda())
    assert dsnq.debug_status() == 0
    dsnq.debug_set(inject_flags=1, wait_timeout_ns=20_000_000)
    try:
        dsnq.block_scaled_fp8_gemm(*args)
        assert dsnq.debug_status() == 5          # DSNQ_ERR_TIMEOUT, and the word is cleared
    finally:
        dsnq.debug_set(0, 0)
    assert dsnq.debug_status() == 0
    out = dsnq.block_scaled_fp8_gemm(*args)
    torch.cuda.synchronize()
    check_gemm(out, a.numpy(), sa.numpy(), wc, ws)
