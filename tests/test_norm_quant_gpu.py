"""Parity of the fused dual RMSNorm + per-1x128 FP8 quant kernel (and of the
unfused baseline kernels and the weight-block quantizer) with the fp64 oracle,
through the C ABI, on the workloads of the method: the PR's 4-token case, the
decode sweep on strided split views, prefill with heavy tails, the
long-context stress with all-zero and single-spike groups, hand-derived exact
cases, ragged shapes and guard bytes around every output."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import (assert_bf16_close, assert_codes_close, assert_scales_close, u8, u16)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CANARY8 = 0x5A
CANARY_F = -12288.0          # exact in bf16 and fp32


def oracle_of(lat, rows=None):
    b = [inputs.bits(t) for t in (lat.q, lat.kv)]
    if rows is not None:
        b = [x[rows] for x in b]
    return oracle.fused_dual_rmsnorm_group_quant(b[0], b[1], inputs.bits(lat.gamma_q),
                                                 inputs.bits(lat.gamma_kv), lat.eps)


def to_device(lat):
    """q and kv on the GPU with the same memory shape as on the host."""
    if lat.buf is not None:
        buf = lat.buf.cuda()
        kq, kkv = lat.q.shape[1], lat.kv.shape[1]
        return buf[:, :kq], buf[:, kq:kq + kkv]
    return lat.q.cuda(), lat.kv.cuda()


def run_guarded(q, kv, gq, gkv, eps, layout, pad_ld=0):
    """Runs the fused kernel into outputs embedded in canary-filled buffers and
    checks that nothing outside the outputs was written."""
    M, Kq = q.shape
    Kkv = kv.shape[1]
    G = Kq // 128
    qbuf = torch.full((M + 2, Kq + 16), CANARY8, dtype=torch.uint8, device="cuda")
    q_out = qbuf[1:M + 1, 8:8 + Kq]
    kvbuf = torch.full((M + 2, Kkv + 16), CANARY_F, dtype=torch.bfloat16, device="cuda")
    kv_out = kvbuf[1:M + 1, 8:8 + Kkv]
    if layout == dsnq.ROW_MAJOR:
        ld = G + pad_ld
        sbuf = torch.full((M * ld + 8,), CANARY_F, dtype=torch.float32, device="cuda")
        scale = sbuf[4:4 + M * ld].view(M, ld)[:, :G]
    else:
        ld = M + pad_ld
        sbuf = torch.full((G * ld + 8,), CANARY_F, dtype=torch.float32, device="cuda")
        scale = sbuf[4:4 + G * ld].view(G, ld)[:, :M].t()
    dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, eps, scale_layout=layout,
                                        q_out=q_out, q_scale=scale, kv_out=kv_out)
    torch.cuda.synchronize()
    # canaries
    qb = qbuf.cpu().numpy()
    inner = np.zeros_like(qb, dtype=bool)
    inner[1:M + 1, 8:8 + Kq] = True
    assert np.all(qb[~inner] == CANARY8), "q_fp8 written out of bounds"
    kb = kvbuf.float().cpu().numpy()
    inner = np.zeros_like(kb, dtype=bool)
    inner[1:M + 1, 8:8 + Kkv] = True
    assert np.all(kb[~inner] == CANARY_F), "kv_out written out of bounds"
    sb = sbuf.cpu().numpy()
    mask = np.zeros(sb.shape, dtype=bool)
    if layout == dsnq.ROW_MAJOR:
        for m in range(M):
            mask[4 + m * ld:4 + m * ld + G] = True
    else:
        for g in range(G):
            mask[4 + g * ld:4 + g * ld + M] = True
    assert np.all(sb[~mask] == CANARY_F), "q_scale written out of bounds"
    return u8(q_out), scale.cpu().numpy(), u16(kv_out)


def check_against_oracle(lat, layout, pad_ld=0):
    q, kv = to_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    codes, scale, kv_out = run_guarded(q, kv, gq, gkv, lat.eps, layout, pad_ld)
    o_codes, o_scale, o_kv = oracle_of(lat)
    assert_scales_close(scale, o_scale)
    exact = assert_codes_close(codes, o_codes)
    assert_bf16_close(kv_out, o_kv)
    return exact


@pytest.mark.parametrize("name", ["hand_case_pow2.json", "hand_case_ties.json"])
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_hand_cases_bit_exact(name, layout):
    c = json.load(open(os.path.join(GOLDEN, name)))
    t = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).cuda()
    codes, scale, kv = run_guarded(t(c["q"]), t(c["kv"]), t(c["gamma_q"]), t(c["gamma_kv"]),
                                   c["eps"], layout)
    assert np.array_equal(codes, np.array(c["expected_codes"], dtype=np.uint8))
    s = c["expected_scale"]
    assert np.all(scale == np.float32(s["numerator"] / s["denominator"]))
    assert np.array_equal(kv, np.array(c["expected_kv_bf16_words"], dtype=np.uint16))


@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_pr1_reference_case(layout):
    check_against_oracle(inputs.pr1_ref(0), layout)


@pytest.mark.parametrize("M", [1, 2, 8, 32, 64])
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_decode_sweep_split_views(M, layout):
    lat = inputs.decode_batch(M, seed=1)
    assert lat.q.stride(0) == inputs.ROW
    check_against_oracle(lat, layout)


@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_padded_scale_leading_dimension(layout):
    check_against_oracle(inputs.decode_batch(8, seed=9), layout, pad_ld=3)


def test_strided_split_view_equals_contiguous():
    lat = inputs.decode_batch(33, seed=4)
    q, kv = to_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    a = dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps)
    b = dsnq.fused_dual_rmsnorm_group_quant(q.contiguous(), kv.contiguous(), gq, gkv, lat.eps)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.float8_e4m3fn else x,
                           y.view(torch.uint8) if y.dtype == torch.float8_e4m3fn else y)


def test_row_and_column_major_scales_transpose_bit_exact():
    lat = inputs.decode_batch(64, seed=6)
    q, kv = to_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    c1, s1, k1 = dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="row")
    c2, s2, k2 = dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="col")
    assert s2.stride() == (1, 64)
    assert torch.equal(s1.view(torch.int32), s2.contiguous().view(torch.int32))
    assert torch.equal(c1.view(torch.uint8), c2.view(torch.uint8)) and torch.equal(k1, k2)


def test_prefill_student_t_full_size():
    exact = check_against_oracle(inputs.prefill_batch(8192, seed=2), dsnq.COL_MAJOR)
    assert exact >= 0.9999


def test_long_context_full_size_sampled_rows():
    M = 32768
    lat = inputs.long_context_batch(M, seed=4)
    q, kv = lat.q.cuda(), lat.kv.cuda()
    codes, scale, kv_out = dsnq.fused_dual_rmsnorm_group_quant(
        q, kv, lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps, scale_layout="col")
    # every edge row, plus a seeded sample of the rest
    edge = sorted({0, M - 1} | set(range(0, M, 97)) | set(range(0, M, 89)))
    rng = np.random.default_rng(0)
    rows = np.array(sorted(set(edge) | set(rng.choice(M, 1024, replace=False).tolist())))
    o_codes, o_scale, o_kv = oracle_of(lat, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_scales_close(scale[idx].cpu().numpy(), o_scale)
    assert_codes_close(u8(codes[idx]), o_codes)
    assert_bf16_close(u16(kv_out[idx]), o_kv)
    s = scale.cpu().numpy()
    assert np.all(s[0] == 0) and np.all(s[M - 1] == 0)
    assert np.all(np.isfinite(s))
    for r in range(0, M, 97):
        if r not in (0, M - 1) and r % 89 != 0:
            assert s[r, r % 12] == 0.0


def test_ragged_shapes_and_small_widths():
    g = torch.Generator().manual_seed(3)
    for M, Kq, Kkv in [(3, 256, 72), (5, 128, 8), (130, 1024, 1024), (2, 2048, 2048)]:
        q = torch.randn(M, Kq, generator=g).to(torch.bfloat16)
        kv = torch.randn(M, Kkv, generator=g).to(torch.bfloat16)
        gq, gkv = inputs.gammas(5, Kq, Kkv)
        lat = inputs.Latents(q, kv, gq, gkv)
        check_against_oracle(lat, dsnq.ROW_MAJOR)


@pytest.mark.parametrize("M", [1216, 1217, 3001, 4869])
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_warp_per_row_ragged_row_counts_split_views(M, layout):
    """DSv4 rows at and past the warp-per-row dispatch point (8 rows per SM on
    the 152-SM part), with row counts that leave warps with zero, one or
    several rows and a ragged last row-round, read from strided split views."""
    check_against_oracle(inputs.decode_batch(M, seed=M), layout)


def test_zero_rows_enqueue_nothing():
    q = torch.empty(0, 1536, dtype=torch.bfloat16, device="cuda")
    kv = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1536, dtype=torch.bfloat16, device="cuda")
    out = dsnq.fused_dual_rmsnorm_group_quant(q, kv, g, g[:512], 1e-6)
    assert out[0].shape == (0, 1536)


# ----------------------------------------------------------------- baselines

def test_baseline_dual_rmsnorm_bf16():
    lat = inputs.decode_batch(32, seed=7)
    q, kv = to_device(lat)
    qo, kvo = dsnq.dual_rmsnorm_bf16(q, kv, lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps)
    wq, wkv = oracle.dual_rmsnorm_bf16(*[inputs.bits(t) for t in (lat.q, lat.kv, lat.gamma_q, lat.gamma_kv)],
                                       lat.eps)
    assert_bf16_close(u16(qo), wq)
    assert_bf16_close(u16(kvo), wkv)


@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_baseline_group_quant_bf16(layout):
    x = inputs.prefill_batch(512, seed=8).q
    codes, scale = dsnq.group_quant_bf16(x.cuda(), scale_layout=layout)
    wc, ws = oracle.group_quant_bf16(inputs.bits(x))
    assert_scales_close(scale.cpu().numpy(), ws)
    assert_codes_close(u8(codes), wc)


@pytest.mark.parametrize("M", [8192, 32768])
def test_baseline_large_m_column_major(M):
    """The unfused three-launch sequence at the sizes the bench times it
    (the warp-per-row kernels in their norm-only and quant-only modes):
    dual RMSNorm to bf16, then the per-1x128 quant of the bf16 q, checked
    against the oracle on every row (M=8192) or on a seeded sample plus the
    first and last rows (M=32768)."""
    lat = inputs.prefill_batch(M, seed=13) if M == 8192 else inputs.long_context_batch(M, seed=14)
    q, kv = lat.q.cuda(), lat.kv.cuda()
    qo, kvo = dsnq.dual_rmsnorm_bf16(q, kv, lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps)
    codes, scale = dsnq.group_quant_bf16(qo, scale_layout="col")
    torch.cuda.synchronize()
    rows = np.arange(M) if M == 8192 else np.array(sorted(
        {0, 1, M - 2, M - 1} | set(np.random.default_rng(2).choice(M, 2048, replace=False).tolist())))
    b = [inputs.bits(t[rows]) for t in (lat.q, lat.kv)]
    wq, wkv = oracle.dual_rmsnorm_bf16(b[0], b[1], inputs.bits(lat.gamma_q), inputs.bits(lat.gamma_kv), lat.eps)
    idx = torch.from_numpy(rows).cuda()
    assert_bf16_close(u16(qo[idx]), wq)
    assert_bf16_close(u16(kvo[idx]), wkv)
    # The quant step is checked on the kernel's own bf16 q (its input).
    wc, ws = oracle.group_quant_bf16(u16(qo[idx]))
    assert_scales_close(scale[idx].cpu().numpy(), ws)
    assert_codes_close(u8(codes[idx]), wc)


def test_weight_block_quantizer():
    w = inputs.weight(4096 + 64, 1536, seed=9)          # ragged last block of 64 rows
    codes, sw = dsnq.quantize_weight_block128(w.cuda())
    wc, ws = oracle.quantize_weight_block128(w.numpy())
    assert_scales_close(sw.cpu().numpy(), ws)
    assert_codes_close(u8(codes), wc)


# ------------------------------------------------------- single-latent variant

@pytest.mark.parametrize("M,K", [(1, 1536), (5, 512), (300, 2048), (2048, 1536), (4, 4096)])
@pytest.mark.parametrize("layout", [dsnq.ROW_MAJOR, dsnq.COL_MAJOR])
def test_single_latent_rmsnorm_group_quant(M, K, layout):
    g = torch.Generator().manual_seed(M + K)
    buf = (torch.randn(M, K + 64, generator=g) * 2.0).to(torch.bfloat16)     # rows of a wider buffer
    x = buf[:, :K]
    gamma = (torch.rand(K, generator=g) + 0.5).to(torch.bfloat16)
    codes, scale = dsnq.rmsnorm_group_quant(buf.cuda()[:, :K], gamma.cuda(), 1e-6, scale_layout=layout)
    wc, ws = oracle.rmsnorm_group_quant(inputs.bits(x.contiguous()), inputs.bits(gamma), 1e-6)
    assert_scales_close(scale.cpu().numpy(), ws)
    assert_codes_close(u8(codes), wc)


@pytest.mark.parametrize("M", [16, 4096])
def test_single_latent_zero_rows_and_matches_fused_q_part(M):
    """The q latent alone gives the q part of the dual call bit for bit, with
    few rows (warp-group kernel) and many (warp-per-row kernel)."""
    lat = inputs.decode_batch(M, seed=12)
    q, kv = to_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    c1, s1 = dsnq.rmsnorm_group_quant(q, gq, lat.eps)
    c2, s2, _ = dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps)
    assert torch.equal(c1.view(torch.uint8), c2.view(torch.uint8)) and torch.equal(s1, s2)
    e = torch.empty(0, 1536, dtype=torch.bfloat16, device="cuda")
    assert dsnq.rmsnorm_group_quant(e, gq, 1e-6)[0].shape == (0, 1536)
