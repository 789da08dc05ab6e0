"""The pre-projection in one call: fused dual RMSNorm + per-1x128 quant of
the q latent (kv latent normalized to bf16), then the dual block-scaled GEMM.
For a few decode rows one launch normalizes and quantizes inside the GEMM;
larger batches run the fused norm+quant kernel, then the GEMM.  Checked
against the oracle (codes, scales, kv_out, both products), against the
hand-derived golden cases bit for bit, and the products against the dual
GEMM applied to the codes and scales the same call wrote."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import inputs
from parity import (GEMM_REL_FRO, assert_bf16_close, assert_codes_close, assert_scales_close, bf16_value,
                    rel_fro)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def quantized_weight(N, K, seed, salt=0):
    return oracle.quantize_weight_block128(inputs.weight(N, K, seed=seed, salt=salt).numpy())


def dev(*arrays):
    return [torch.from_numpy(x).cuda() for x in arrays]


def on_device(lat):
    if lat.buf is not None:                       # split views of one [M, 2112] buffer
        buf = lat.buf.cuda()
        return buf[:, :inputs.KQ], buf[:, inputs.KQ:inputs.KQ + inputs.KKV]
    return lat.q.cuda(), lat.kv.cuda()


def run(q, kv, gq, gkv, eps, w, with_q_outputs=True):
    M, Kq = q.shape
    qf = torch.empty(M, Kq, dtype=torch.float8_e4m3fn, device="cuda") if with_q_outputs else None
    qs = dsnq.empty_scales(M, Kq // 128, "col", "cuda") if with_q_outputs else None
    return dsnq.fused_norm_quant_gemm_dual(q, kv, gq, gkv, eps, *w, q_fp8=qf, q_scale=qs)


@pytest.mark.parametrize("M", [1, 2, 5, 6, 7, 64, 300])
def test_matches_oracle(M):
    lat = inputs.decode_batch(M, seed=70 + M) if M <= 64 else inputs.full_path_batch(M, seed=71)
    q, kv = on_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    w1, s1 = quantized_weight(1024, inputs.KQ, seed=72)
    w2, s2 = quantized_weight(512, inputs.KQ, seed=73)
    W = dev(w1, s1, w2, s2)
    o1, o2, kvo, qf, qs = run(q, kv, gq, gkv, lat.eps, W)
    torch.cuda.synchronize()
    codes, scale, kv_bits = oracle.fused_dual_rmsnorm_group_quant(
        inputs.bits(lat.q), inputs.bits(lat.kv), inputs.bits(lat.gamma_q), inputs.bits(lat.gamma_kv), lat.eps)
    assert_codes_close(qf.view(torch.uint8).cpu().numpy(), codes)
    assert_scales_close(qs.cpu().numpy(), scale)
    assert_bf16_close(kvo.view(torch.int16).cpu().numpy().view(np.uint16), kv_bits)
    for out, wc, ws in ((o1, w1, s1), (o2, w2, s2)):
        ref = oracle.block_scaled_gemm(codes, scale, wc, ws)
        assert rel_fro(bf16_value(out), ref) <= GEMM_REL_FRO
    # The products are those of the dual GEMM on the codes and scales written.
    t1, t2 = dsnq.block_scaled_fp8_gemm_dual(qf, qs, *W)
    assert torch.equal(o1, t1) and torch.equal(o2, t2)


@pytest.mark.parametrize("M,Kq", [(1, 1408), (3, 1408), (6, 1408), (1, 2048), (2, 2048), (5, 512), (8, 512),
                                  (8, 1280), (7, 1024)])
def test_one_launch_other_widths(M, Kq):
    """The one-launch route at other q widths: an odd number of K blocks (the
    last 256-column unit half past the row), the widest row it takes (eight
    units), and a narrow one; one to eight rows (all of the resident operand's
    rows) spread over the quantizer warps."""
    assert dsnq.fused_quant_fits(M, Kq)
    g = torch.Generator().manual_seed(90 + M + Kq)
    q = (torch.randn(M, Kq, generator=g) * 2.0).to(torch.bfloat16)
    kv = torch.randn(M, 512, generator=g).to(torch.bfloat16)
    gq, gkv = inputs.gammas(91, Kq, 512)
    w1, s1 = quantized_weight(384, Kq, seed=92)
    w2, s2 = quantized_weight(256, Kq, seed=93)
    W = dev(w1, s1, w2, s2)
    o1, o2, kvo, qf, qs = run(q.cuda(), kv.cuda(), gq.cuda(), gkv.cuda(), 1e-6, W)
    torch.cuda.synchronize()
    codes, scale, kv_bits = oracle.fused_dual_rmsnorm_group_quant(
        inputs.bits(q), inputs.bits(kv), inputs.bits(gq), inputs.bits(gkv), 1e-6)
    assert_codes_close(qf.view(torch.uint8).cpu().numpy(), codes)
    assert_scales_close(qs.cpu().numpy(), scale)
    assert_bf16_close(kvo.view(torch.int16).cpu().numpy().view(np.uint16), kv_bits)
    for out, wc, ws in ((o1, w1, s1), (o2, w2, s2)):
        ref = oracle.block_scaled_gemm(codes, scale, wc, ws)
        assert rel_fro(bf16_value(out), ref) <= GEMM_REL_FRO
    t1, t2 = dsnq.block_scaled_fp8_gemm_dual(qf, qs, *W)
    assert torch.equal(o1, t1) and torch.equal(o2, t2)


def test_one_launch_without_q_outputs():
    lat = inputs.decode_batch(3, seed=80)
    q, kv = on_device(lat)
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    wa, swa = quantized_weight(inputs.N_ATTN, inputs.KQ, seed=0, salt=1)
    wi, swi = quantized_weight(inputs.N_IDX, inputs.KQ, seed=0, salt=2)
    W = dev(wa, swa, wi, swi)
    a1, a2, akv, qf, qs = run(q, kv, gq, gkv, lat.eps, W, with_q_outputs=False)
    assert qf is None and qs is None
    b1, b2, bkv, _, _ = run(q, kv, gq, gkv, lat.eps, W)
    assert torch.equal(a1, b1) and torch.equal(a2, b2) and torch.equal(akv, bkv)


@pytest.mark.parametrize("name", ["hand_case_pow2.json", "hand_case_ties.json"])
def test_hand_cases_bit_exact(name):
    """Golden rows (M=1, Kq=128) through the one-launch path."""
    c = json.load(open(os.path.join(GOLDEN, name)))
    t = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).cuda()
    q, kv = t(c["q"]), t(c["kv"])
    w1, s1 = quantized_weight(16, 128, seed=90)
    W = dev(w1, s1, w1, s1)
    o1, _, kvo, qf, qs = run(q, kv, t(c["gamma_q"]), t(c["gamma_kv"]), c["eps"], W)
    torch.cuda.synchronize()
    assert np.array_equal(qf.view(torch.uint8).cpu().numpy(), np.array(c["expected_codes"], dtype=np.uint8))
    s = c["expected_scale"]
    assert np.all(qs.cpu().numpy() == np.float32(s["numerator"] / s["denominator"]))
    assert np.array_equal(kvo.view(torch.int16).cpu().numpy().view(np.uint16),
                          np.array(c["expected_kv_bf16_words"], dtype=np.uint16))
    ref = oracle.block_scaled_gemm(qf.view(torch.uint8).cpu().numpy(), qs.cpu().numpy(), w1, s1)
    assert rel_fro(bf16_value(o1), ref) <= GEMM_REL_FRO
