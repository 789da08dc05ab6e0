"""Pins of the fp64 CPU oracle against facts that do not come from the oracle:
the E4M3FN and bf16 formats (exhaustive code tables, torch's casts as a
library special case), torch's float64 rms_norm and matmul, closed forms,
hand-derived cases (tests/golden/) and invariants of the method.  CPU only."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from gemm_dsnq_dual_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v) -> np.ndarray:
    return inputs.bits(torch.as_tensor(np.asarray(v, dtype=np.float32)).to(torch.bfloat16))


# ------------------------------------------------------------------ formats

def test_e4m3_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254              # only S.1111.111 are NaN
    assert np.array_equal(oracle.e4m3_encode(vals[finite]), codes[finite])


def test_e4m3_table_landmarks():
    d = oracle.e4m3_decode
    assert d(np.uint8(0x7E)) == 448.0          # max finite
    assert d(np.uint8(0x08)) == 2.0 ** -6      # min normal
    assert d(np.uint8(0x01)) == 2.0 ** -9      # min subnormal
    assert d(np.uint8(0x38)) == 1.0            # exponent bias 7
    assert d(np.uint8(0xB8)) == -1.0
    assert np.isnan(d(np.uint8(0x7F))) and np.isnan(d(np.uint8(0xFF)))


def test_e4m3_midpoints_round_to_even():
    codes = np.arange(0x00, 0x7E, dtype=np.uint8)       # adjacent finite pairs (c, c+1)
    lo = oracle.e4m3_decode(codes)
    hi = oracle.e4m3_decode(codes + 1)
    mid = (lo + hi) / 2
    even = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(mid), even)
    assert np.array_equal(oracle.e4m3_encode(-mid), even | 0x80)
    # just off the midpoint goes to the nearer code
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, 0)), codes)
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, 1e9)), codes + 1)


def test_e4m3_saturates_and_signed_zero():
    assert list(oracle.e4m3_encode(np.array([448.0, 449.0, 464.0, 1e6, 1e300]))) == [0x7E] * 5
    assert list(oracle.e4m3_encode(np.array([-448.0, -500.0, -1e30]))) == [0xFE] * 3
    assert oracle.e4m3_encode(np.array([-1e-9]))[0] == 0x80
    assert oracle.e4m3_encode(np.array([-0.0]))[0] == 0x80
    assert oracle.e4m3_encode(np.array([0.0]))[0] == 0x00


def test_e4m3_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(200_000, generator=g) * torch.exp2(torch.randint(-14, 9, (200_000,), generator=g).float())
    x = x[x.abs() <= 448.0]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.double().numpy())
    assert np.array_equal(got, want)


def test_bf16_matches_torch_cast_from_fp32():
    g = torch.Generator().manual_seed(12)
    x = torch.randn(200_000, generator=g) * torch.exp2(torch.randint(-40, 40, (200_000,), generator=g).float())
    want = inputs.bits(x.to(torch.bfloat16))
    got = oracle.f64_to_bf16_bits(x.double().numpy())
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.bf16_bits_to_f64(want), x.to(torch.bfloat16).double().numpy())


def test_bf16_rounds_once_from_fp64():
    # 1 + 2^-8 + 2^-30: fp32 would round it to the bf16 midpoint 1 + 2^-8 and
    # then to even (1.0); one rounding from fp64 gives the upper neighbour.
    v = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(v))[0] == 1.0 + 2.0 ** -7
    assert oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8])))[0] == 1.0


# ------------------------------------------------------------------ RMSNorm + quant

def test_rmsnorm_matches_torch_float64():
    lat = inputs.pr1_ref(0)
    x = torch.from_numpy(oracle.bf16_bits_to_f64(inputs.bits(lat.q)))
    gq = torch.from_numpy(oracle.bf16_bits_to_f64(inputs.bits(lat.gamma_q)))
    eps = float(np.float32(lat.eps))
    want = torch.nn.functional.rms_norm(x, (x.shape[1],), weight=gq, eps=eps).numpy()
    xq, _ = oracle.normalized_latents(inputs.bits(lat.q), inputs.bits(lat.kv),
                                      inputs.bits(lat.gamma_q), inputs.bits(lat.gamma_kv), lat.eps)
    np.testing.assert_allclose(xq, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("c", [0.75, -3.0, 1e-3])
def test_constant_row_closed_form(c):
    Kq, Kkv, eps = 256, 16, 1e-6
    q = bf16(np.full((2, Kq), c))
    kv = bf16(np.full((2, Kkv), c))
    cb = float(oracle.bf16_bits_to_f64(q)[0, 0])
    e = float(np.float32(eps))
    xhat = cb / np.sqrt(cb * cb + e)
    codes, scale, kv_out = oracle.fused_dual_rmsnorm_group_quant(q, kv, bf16(np.ones(Kq)), bf16(np.ones(Kkv)), eps)
    assert np.all(codes == (0xFE if c < 0 else 0x7E))
    assert np.all(scale == np.float32(abs(xhat)) / np.float32(448.0))
    assert np.all(oracle.bf16_bits_to_f64(kv_out) == float(torch.tensor(xhat, dtype=torch.float64).to(torch.bfloat16)))


def test_single_spike_group_and_zero_group():
    Kq, Kkv = 384, 8
    row = np.random.default_rng(0).standard_normal(Kq)
    row[128:256] = 0.0
    row[128 + 37] = -1000.0               # group 1: one spike, rest zero
    row[256:384] = 0.0                     # group 2: all zero
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(
        bf16(row[None]), bf16(np.ones((1, Kkv))), bf16(np.ones(Kq)), bf16(np.ones(Kkv)), 1e-6)
    g1 = codes[0, 128:256]
    assert g1[37] == 0xFE and np.all(np.delete(g1, 37) == 0)
    assert scale[0, 2] == 0.0 and np.all(codes[0, 256:] == 0)
    assert scale[0, 1] > 0


def test_all_zero_row_is_zero_not_nan():
    codes, scale, kv = oracle.fused_dual_rmsnorm_group_quant(
        bf16(np.zeros((1, 256))), bf16(np.zeros((1, 64))), bf16(np.ones(256)), bf16(np.ones(64)), 1e-6)
    assert np.all(codes == 0) and np.all(scale == 0) and np.all(kv == 0)


@pytest.mark.parametrize("name", ["hand_case_pow2.json", "hand_case_ties.json"])
def test_hand_cases(name):
    c = json.load(open(os.path.join(GOLDEN, name)))
    codes, scale, kv = oracle.fused_dual_rmsnorm_group_quant(
        bf16(c["q"]), bf16(c["kv"]), bf16(c["gamma_q"]), bf16(c["gamma_kv"]), c["eps"])
    assert np.array_equal(codes, np.array(c["expected_codes"], dtype=np.uint8))
    s = c["expected_scale"]
    assert np.all(scale == np.float32(s["numerator"] / s["denominator"]))
    assert np.array_equal(kv, np.array(c["expected_kv_bf16_words"], dtype=np.uint16))


def _decode_batch_oracle(M, seed=1):
    lat = inputs.decode_batch(M, seed)
    xq, _ = oracle.normalized_latents(inputs.bits(lat.q), inputs.bits(lat.kv), inputs.bits(lat.gamma_q),
                                      inputs.bits(lat.gamma_kv), lat.eps)
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(
        inputs.bits(lat.q), inputs.bits(lat.kv), inputs.bits(lat.gamma_q), inputs.bits(lat.gamma_kv), lat.eps)
    return xq, codes, scale


def test_quant_invariants_half_ulp_and_amax():
    xq, codes, scale = _decode_batch_oracle(32)
    M, K = xq.shape
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    q = xq / s
    deq = oracle.e4m3_decode(codes)
    # half an E4M3 ULP of the quotient: spacing 2^(e-3) in binade e, 2^-9 below
    # 2^-6; the quotient itself is an fp32 value, hence the 2^-23 relative slack
    e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
    half_ulp = 0.5 * 2.0 ** (e - 3)
    assert np.all(np.abs(deq - q) <= half_ulp + np.abs(q) * 2.0 ** -23)
    # amax element of every group maps to +-448
    g = np.abs(xq).reshape(M, K // 128, 128)
    arg = g.argmax(axis=-1)
    top = np.take_along_axis(codes.reshape(M, K // 128, 128), arg[..., None], -1)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))


def test_quant_decision_is_taken_on_the_fp32_quotient():
    # Documents the reading (not a pin): with amax = 3 the scale fp32(3/448)
    # is inexact, so a quotient that is an exact E4M3 midpoint in real
    # arithmetic may fall on either side of it in fp64; the code is the E4M3
    # rounding of the fp32 quotient fp32(x / scale).
    x = np.zeros((1, 128), np.float64)
    x[0, 0] = 3.0
    x[0, 1:] = np.linspace(-3, 3, 127).astype(np.float32).astype(np.float64)
    codes, scale = oracle.group_quant_f64(x)
    s = np.float32(3.0) / np.float32(448.0)
    q32 = x.astype(np.float32) / s
    assert scale[0, 0] == s
    assert np.array_equal(codes, oracle.e4m3_encode(q32.astype(np.float64)))
    assert codes[0, 0] == 0x7E


def test_row_and_column_major_scales_are_transposes():
    _, _, scale = _decode_batch_oracle(8)
    M, G = scale.shape
    rm = oracle.store_scales(scale, oracle.SCALE_ROW_MAJOR)
    cm = oracle.store_scales(scale, oracle.SCALE_COL_MAJOR)
    assert np.array_equal(rm.reshape(M, G).T.view(np.uint32), cm.reshape(G, M).view(np.uint32))
    assert np.array_equal(oracle.load_scales(cm, M, G, oracle.SCALE_COL_MAJOR), scale)
    # padded leading dimensions leave the gaps untouched
    cm2 = oracle.store_scales(scale, oracle.SCALE_COL_MAJOR, ld=M + 3)
    assert np.array_equal(oracle.load_scales(cm2, M, G, oracle.SCALE_COL_MAJOR, ld=M + 3), scale)
    assert np.isnan(cm2[M])


def test_fused_single_rounding_is_at_least_as_accurate():
    # The fused path quantizes the fp32/fp64 normalized values; the unfused
    # one rounds them to bf16 first (PR #53540, Purpose: single rounding,
    # equivalent-or-better precision).  Compare in the dequantized domain.
    lat = inputs.prefill_batch(256, seed=5)
    b = [inputs.bits(t) for t in (lat.q, lat.kv, lat.gamma_q, lat.gamma_kv)]
    xq, _ = oracle.normalized_latents(*b, lat.eps)
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(*b, lat.eps)
    qb, _ = oracle.dual_rmsnorm_bf16(*b, lat.eps)
    codes_u, scale_u = oracle.group_quant_bf16(qb)
    err_f = np.linalg.norm(oracle.dequantize_activation(codes, scale) - xq)
    err_u = np.linalg.norm(oracle.dequantize_activation(codes_u, scale_u) - xq)
    assert err_f <= err_u
    assert (codes != codes_u).mean() > 0.001     # the two really differ


# ------------------------------------------------------------------ GEMM

def test_bf16_group_quant_matches_torch_fp32_quotient_and_cast():
    """The quant of bf16 activations (baseline step 2, and the GEMM on bf16
    activations): scale = fp32 division amax / 448 and code = torch's e4m3
    cast of the fp32 quotient x / scale, computed entirely by torch."""
    g = torch.Generator().manual_seed(12)
    x = (torch.randn(64, 1536, generator=g) * torch.exp2(torch.randint(-6, 6, (64, 1, 1536 // 128), generator=g)
                                                          .float().repeat_interleave(128, dim=2).squeeze(1)))
    x[3] = 0.0                                                   # an all-zero row
    xb = x.to(torch.bfloat16)
    codes, scale = oracle.group_quant_bf16(inputs.bits(xb))
    x32 = xb.float().view(64, 12, 128)
    amax = x32.abs().amax(dim=2)
    s32 = amax / torch.tensor(448.0)                             # IEEE fp32 division
    q = torch.where(s32[..., None] > 0, x32 / s32[..., None].clamp_min(torch.finfo(torch.float32).tiny), x32 * 0)
    want_codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(64, 1536).numpy()
    assert np.array_equal(scale, s32.numpy())
    assert np.array_equal(codes, want_codes)


def test_weight_block_quant_properties():
    w = inputs.weight(300, 256, seed=1).numpy()       # ragged N: 3 blocks, last 44 rows
    codes, sw = oracle.quantize_weight_block128(w)
    assert sw.shape == (3, 2)
    for i in range(3):
        for j in range(2):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert sw[i, j] == np.abs(blk).max() / np.float32(448.0)
            r, c = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            assert codes[i * 128 + r, j * 128 + c] in (0x7E, 0xFE)
    deq = oracle.dequantize_weight(codes, sw)
    rel = np.abs(deq - w) / np.repeat(np.repeat(sw.astype(np.float64), 128, 0)[:300], 128, 1)
    assert rel.max() <= 0.5 * 32 * (1 + 1e-9)      # half ULP at the top binade (spacing 32)


def test_gemm_matches_torch_matmul_float64():
    a, sa = inputs.random_codes_and_scales(37, 512, seed=3)
    w = inputs.weight(272, 512, seed=4).numpy()
    wc, sw = oracle.quantize_weight_block128(w)
    got = oracle.block_scaled_gemm(a.numpy(), sa.numpy(), wc, sw)
    A = torch.from_numpy(oracle.e4m3_decode(a.numpy())) * torch.from_numpy(sa.numpy().astype(np.float64)).repeat_interleave(128, 1)
    W = torch.from_numpy(oracle.e4m3_decode(wc)) * torch.from_numpy(sw.astype(np.float64)).repeat_interleave(128, 0)[:272].repeat_interleave(128, 1)
    np.testing.assert_allclose(got, (A @ W.T).numpy(), rtol=1e-12, atol=1e-12)


def test_gemm_exact_on_small_integers():
    # Codes of small integers with unit scales: every product and sum is an
    # integer well inside fp64, so the result is exact.
    rng = np.random.default_rng(5)
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, -1, -2, -3, -4, -8])
    ai = rng.choice(ints, size=(5, 256))
    wi = rng.choice(ints, size=(144, 256))
    a = oracle.e4m3_encode(ai.astype(np.float64))
    w = oracle.e4m3_encode(wi.astype(np.float64))
    got = oracle.block_scaled_gemm(a, np.ones((5, 2), np.float32), w, np.ones((2, 2), np.float32))
    want = np.array([[int(np.dot(ai[m].astype(object), wi[n].astype(object))) for n in range(144)] for m in range(5)])
    assert np.array_equal(got, want.astype(np.float64))


def test_gemm_bruteforce_triple_loop():
    a, sa = inputs.random_codes_and_scales(3, 256, seed=7)
    w = inputs.weight(130, 256, seed=8).numpy()[:, :]
    wc, sw = oracle.quantize_weight_block128(np.pad(w, ((0, 14), (0, 0))))   # N=144, multiple of 16
    a, sa = a.numpy(), sa.numpy()
    dec_a, dec_w = oracle.e4m3_decode(a), oracle.e4m3_decode(wc)
    got = oracle.block_scaled_gemm(a, sa, wc, sw)
    for m in range(3):
        for n in range(0, 144, 7):
            acc = 0.0
            for kb in range(2):
                part = 0.0
                for k in range(kb * 128, (kb + 1) * 128):
                    part += dec_a[m, k] * dec_w[n, k]
                acc += float(sa[m, kb]) * float(sw[n // 128, kb]) * part
            assert abs(acc - got[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_single_latent_is_the_q_part_of_the_fused_op():
    """The single-latent op is the fused op's q computation on its own: same
    codes and scales for the same latent, whatever the kv latent is."""
    rng = np.random.default_rng(11)
    q = oracle.f64_to_bf16_bits(rng.standard_normal((6, 512)) * 3.0)
    kv = oracle.f64_to_bf16_bits(rng.standard_normal((6, 64)))
    gq = oracle.f64_to_bf16_bits(rng.uniform(0.5, 1.5, 512))
    gkv = oracle.f64_to_bf16_bits(rng.uniform(0.5, 1.5, 64))
    c1, s1 = oracle.rmsnorm_group_quant(q, gq, 1e-6)
    c2, s2, _ = oracle.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, 1e-6)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    # constant row: every code is +-448 and the scale is |x_hat| / 448
    const = oracle.f64_to_bf16_bits(np.full((1, 256), 2.0))
    ones = oracle.f64_to_bf16_bits(np.ones(256))
    c, s = oracle.rmsnorm_group_quant(const, ones, 0.0)
    assert np.all(c == 0x7E) and np.allclose(s, np.float32(1.0) / np.float32(448.0))


def _plain_fp64_quotient_codes(q_bits, kv_bits, gq_bits, gkv_bits, eps, group=128):
    """The quant step by its plain definition, all in fp64: x_hat from the
    fp64 RMSNorm (not rounded to fp32), amax of x_hat, the scale stored as
    fp32(amax / 448), and code = e4m3(x_hat / scale) with the quotient left in
    fp64.  Written here from the definition, independently of the oracle's
    fp32-quotient reading."""
    eps = float(np.float32(eps))
    x = oracle.bf16_bits_to_f64(q_bits)
    ms = np.mean(x * x, axis=1, keepdims=True)
    xhat = x / np.sqrt(ms + eps) * oracle.bf16_bits_to_f64(gq_bits)
    M, K = xhat.shape
    g = xhat.reshape(M, K // group, group)
    s = (np.max(np.abs(g), axis=-1) / 448.0).astype(np.float32).astype(np.float64)[..., None]
    quot = np.where(s > 0, g / np.where(s > 0, s, 1.0), g * 0.0)
    return oracle.e4m3_encode(quot).reshape(M, K)


@pytest.mark.parametrize("workload", ["decode", "prefill", "long_context"])
def test_fp32_quotient_reading_stays_within_tolerance_of_the_plain_definition(workload):
    """The oracle takes the quantize decision on the fp32 quotient (the
    pages' "reads the fp32 accumulator").  Against the same step taken
    entirely in fp64 (the plain definition, a different but well-defined
    code), its codes are within one E4M3 step and at least 99.9% identical
    on the workloads' inputs: the stated tolerance holds against the plain
    definition too, not only against the reading."""
    from parity import CODE_EXACT_MIN, code_ordinal
    if workload == "decode":
        lat = inputs.decode_batch(64, seed=1)
        rows = slice(None)
    elif workload == "prefill":
        lat = inputs.prefill_batch(8192, seed=2)
        rows = np.random.default_rng(5).choice(8192, 2048, replace=False)
    else:
        lat = inputs.long_context_batch(32768, seed=4)
        M = 32768
        edge = {0, M - 1} | set(range(0, M, 97)) | set(range(0, M, 89))
        rows = np.array(sorted(edge | set(np.random.default_rng(6).choice(M, 1024, replace=False).tolist())))
    b = [inputs.bits(t.contiguous()) for t in (lat.q, lat.kv)]
    qb, kvb = b[0][rows], b[1][rows]
    gq, gkv = inputs.bits(lat.gamma_q), inputs.bits(lat.gamma_kv)
    codes, _, _ = oracle.fused_dual_rmsnorm_group_quant(qb, kvb, gq, gkv, lat.eps)
    plain = _plain_fp64_quotient_codes(qb, kvb, gq, gkv, lat.eps)
    d = np.abs(code_ordinal(codes) - code_ordinal(plain))
    assert d.max() <= 1
    assert (d == 0).mean() >= CODE_EXACT_MIN
