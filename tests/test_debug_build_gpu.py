"""The debug build (libdsnq_debug.so, compiled with DSNQ_DEBUG): every
kernel checks the indices of its memory accesses against the extents its
arguments describe.  One small case per kernel runs under it, its results are
checked against the release build bit for bit, and the device status words
must report no failed check; the reporting path itself is exercised with the
hook that records one deliberate failed check guarding no access."""

import numpy as np
import pytest
import torch

import oracle
import gemm_dsnq_dual_gb300 as dsnq
from gemm_dsnq_dual_gb300 import _native, inputs

pytestmark = pytest.mark.gpu
OK, BOUNDS = 0, 6


@pytest.fixture(scope="module")
def libs():
    release = _native.LIB_PATH
    yield release, _native.DEBUG_LIB_PATH
    _native.use_library(release)


def run_every_kernel():
    """One small call of each kernel; returns every output tensor."""
    outs = []
    lat = inputs.decode_batch(4, seed=31)                     # warp-group-per-row kernel, split views
    buf = lat.buf.cuda()
    gq, gkv = lat.gamma_q.cuda(), lat.gamma_kv.cuda()
    outs += dsnq.fused_dual_rmsnorm_group_quant(buf[:, :1536], buf[:, 1536:2048], gq, gkv, lat.eps, scale_layout="col")
    big = inputs.full_path_batch(1536, seed=32)               # DSv4 warp-per-row kernel (M >= 8 x SMs)
    q, kv = big.q.cuda(), big.kv.cuda()
    outs += dsnq.fused_dual_rmsnorm_group_quant(q, kv, gq, gkv, lat.eps, scale_layout="row")
    outs += dsnq.rmsnorm_group_quant(q[:5], gq, lat.eps)      # single latent
    qb, kvb = dsnq.dual_rmsnorm_bf16(q, kv, gq, gkv, lat.eps)  # unfused baseline, warp-per-row modes
    outs += [qb, kvb]
    outs += dsnq.group_quant_bf16(qb, scale_layout="col")
    outs += dsnq.group_quant_bf16(qb[:7])                     # warp-group mode
    outs += dsnq.quantize_weight_block128(inputs.weight(300, 1536, seed=33).cuda())
    w1, s1 = dsnq.quantize_weight_block128(inputs.weight(512, 1536, seed=34).cuda())
    w2, s2 = dsnq.quantize_weight_block128(inputs.weight(256, 1536, seed=35).cuda())
    for M in (3, 40, 100, 300):                               # decode, decode BN=64, 128x128 tiles, CTA pair
        a8, sa = dsnq.fused_dual_rmsnorm_group_quant(q[:M], kv[:M], gq, gkv, lat.eps, scale_layout="col")[:2]
        outs += dsnq.block_scaled_fp8_gemm_dual(a8, sa, w1, s1, w2, s2)
    xa = inputs.activations_bf16(2, 1536, seed=36).cuda()
    outs += dsnq.block_scaled_fp8_gemm_dual_bf16a(xa, w1, s1, w2, s2)         # quantized in the prologue
    outs += dsnq.fused_norm_quant_gemm_dual(buf[:2, :1536], buf[:2, 1536:2048], gq, gkv, lat.eps, w1, s1, w2, s2)[:3]
    torch.cuda.synchronize()
    return outs


def as_bits(t):
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return t.contiguous().view(torch.uint8)
    return t.contiguous().view(torch.int16) if t.element_size() == 2 else t.contiguous().view(torch.int32)


def test_every_kernel_passes_its_index_checks_and_matches_the_release_build(libs):
    release, debug = libs
    _native.use_library(release)
    want = run_every_kernel()
    _native.use_library(debug)
    assert _native.lib().dsnq_debug_build() == 1
    assert dsnq.debug_status() == OK
    got = run_every_kernel()
    assert dsnq.debug_status() == OK                          # no check failed
    assert len(got) == len(want)
    for g, w in zip(got, want):
        assert torch.equal(as_bits(g), as_bits(w))


def test_a_failed_check_is_reported_and_cleared(libs):
    """The hook records one failed check per launch without any access
    attached; dsnq_debug_status reports it once and clears the words."""
    _, debug = libs
    _native.use_library(debug)
    lat = inputs.pr1_ref(0)
    args = (lat.q.cuda(), lat.kv.cuda(), lat.gamma_q.cuda(), lat.gamma_kv.cuda(), lat.eps)
    ref = dsnq.fused_dual_rmsnorm_group_quant(*args)
    assert dsnq.debug_status() == OK
    dsnq.debug_set(inject_flags=2)
    try:
        got = dsnq.fused_dual_rmsnorm_group_quant(*args)
        assert dsnq.debug_status() == BOUNDS
    finally:
        dsnq.debug_set(0, 0)
    assert dsnq.debug_status() == OK
    for g, w in zip(got, ref):                                # the computation itself is unaffected
        assert torch.equal(as_bits(g), as_bits(w))
    codes, scale, _ = oracle.fused_dual_rmsnorm_group_quant(*[inputs.bits(t) for t in
                                                             (lat.q, lat.kv, lat.gamma_q, lat.gamma_kv)], lat.eps)
    assert np.array_equal(scale, got[1].cpu().numpy()) or np.allclose(scale, got[1].cpu().numpy(), rtol=1e-6)
