"""The C ABI without a GPU: the library loads, exports every symbol that
include/dsnq.h declares, and rejects bad arguments on the host before it
would enqueue anything (these calls never reach the CUDA runtime)."""

import ctypes as C
import os
import re

import pytest

from gemm_dsnq_dual_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsnq.h")

OK, INVALID, MISALIGNED, UNSUPPORTED = 0, 1, 2, 3
A = 0x10000          # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        build.build()
    return _native.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(dsnq_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(_native.SIGNATURES)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_debug_build_exports_the_same_symbols():
    """The debug build (device index checks) has the same C ABI."""
    import ctypes
    if not os.path.exists(_native.DEBUG_LIB_PATH):
        build.build()
    h = ctypes.CDLL(_native.DEBUG_LIB_PATH)
    for name in declared_functions():
        assert hasattr(h, name), name
    h.dsnq_debug_build.restype = ctypes.c_int32
    assert h.dsnq_debug_build() == 1


def test_status_strings_and_version(lib):
    for s, name in _native.STATUS_NAMES.items():
        assert lib.dsnq_status_string(s).decode() == name
    assert lib.dsnq_status_string(99).decode() == "DSNQ_ERR_UNKNOWN"
    assert lib.dsnq_version() >= 100
    assert lib.dsnq_debug_build() == 0          # the release build


def test_quant_output_sizes(lib):
    n, ld = C.c_int64(), C.c_int64()
    assert lib.dsnq_quant_output_sizes(7, 1536, 128, 0, C.byref(n), C.byref(ld)) == OK
    assert (n.value, ld.value) == (7 * 12, 12)
    assert lib.dsnq_quant_output_sizes(7, 1536, 128, 1, C.byref(n), C.byref(ld)) == OK
    assert (n.value, ld.value) == (7 * 12, 7)
    assert lib.dsnq_quant_output_sizes(7, 1536, 64, 0, None, None) == UNSUPPORTED
    assert lib.dsnq_quant_output_sizes(7, 1500, 128, 0, None, None) == UNSUPPORTED
    assert lib.dsnq_quant_output_sizes(-1, 1536, 128, 0, None, None) == INVALID
    assert lib.dsnq_quant_output_sizes(7, 1536, 128, 5, None, None) == INVALID


def fused(lib, **kw):
    a = dict(M=4, Kq=1536, Kkv=512, q=A, ldq=2112, kv=A + 3072, ldkv=2112, gq=A, gkv=A, eps=1e-6,
             group=128, qo=A, ldqo=1536, qs=A, layout=0, lds=0, kvo=A, ldkvo=512)
    a.update(kw)
    return lib.dsnq_fused_dual_rmsnorm_group_quant(
        a["M"], a["Kq"], a["Kkv"], a["q"], a["ldq"], a["kv"], a["ldkv"], a["gq"], a["gkv"], a["eps"],
        a["group"], a["qo"], a["ldqo"], a["qs"], a["layout"], a["lds"], a["kvo"], a["ldkvo"], None)


def test_fused_argument_checks(lib):
    assert fused(lib, M=0) == OK                     # no rows: nothing enqueued
    assert fused(lib, M=0, q=None, kv=None, qo=None, qs=None, kvo=None) == OK
    assert fused(lib, M=-1) == INVALID
    assert fused(lib, q=None) == INVALID
    assert fused(lib, qs=None) == INVALID
    assert fused(lib, ldq=1000) == INVALID           # ld < width
    assert fused(lib, layout=7) == INVALID
    assert fused(lib, layout=1, lds=3) == INVALID    # column-major ld < M
    assert fused(lib, layout=0, lds=11) == INVALID   # row-major ld < G
    assert fused(lib, eps=-1.0) == INVALID
    assert fused(lib, eps=float("nan")) == INVALID
    assert fused(lib, group=64) == UNSUPPORTED
    assert fused(lib, Kq=1500) == UNSUPPORTED
    assert fused(lib, Kkv=500) == UNSUPPORTED
    assert fused(lib, Kq=4096, Kkv=512, ldq=4608, ldkv=4608, ldqo=4096) == UNSUPPORTED  # > 4 chunks per thread
    assert fused(lib, q=A + 8) == MISALIGNED
    assert fused(lib, ldq=2100) == MISALIGNED
    assert fused(lib, kvo=A + 4) == MISALIGNED
    assert fused(lib, qo=A + 4) == MISALIGNED
    assert fused(lib, qs=A + 2) == MISALIGNED


def gemm(lib, **kw):
    a = dict(M=0, N=512, K=1536, a=A, lda=1536, sa=A, lay=0, lds=0, w=A, ldw=1536, sw=A, ldsw=12,
             o=A, ldo=512)
    a.update(kw)
    return lib.dsnq_block_scaled_fp8_gemm(a["M"], a["N"], a["K"], a["a"], a["lda"], a["sa"], a["lay"], a["lds"],
                                          a["w"], a["ldw"], a["sw"], a["ldsw"], a["o"], a["ldo"], None)


def test_gemm_argument_checks(lib):
    assert gemm(lib) == OK                            # M == 0
    assert gemm(lib, M=4, N=0) == OK
    assert gemm(lib, a=None, sa=None) == OK          # empty activations may be NULL
    assert gemm(lib, M=-1) == INVALID
    assert gemm(lib, M=4, a=None) == INVALID
    assert gemm(lib, K=1000, lda=1000, ldw=1000) == UNSUPPORTED
    assert gemm(lib, M=4, N=520, ldo=520) == UNSUPPORTED   # N % 16
    assert gemm(lib, M=4, lda=1000) == INVALID
    assert gemm(lib, M=4, ldsw=11) == INVALID
    assert gemm(lib, M=4, a=A + 8) == MISALIGNED
    assert gemm(lib, M=4, lda=1544) == MISALIGNED
    assert gemm(lib, M=4, o=A + 2) == MISALIGNED
    assert gemm(lib, lay=3) == INVALID


def test_dual_and_helpers_argument_checks(lib):
    f = lib.dsnq_block_scaled_fp8_gemm_dual
    assert f(0, 1536, A, 1536, A, 0, 0, 512, A, 1536, A, 12, A, 512, 256, A, 1536, A, 12, A, 256, None) == OK
    assert f(4, 1536, A, 1536, A, 0, 0, 512, A, 1536, A, 12, A, 512, 256, A + 1, 1536, A, 12, A, 256, None) == MISALIGNED
    assert f(4, 1536, A, 1536, A, 0, 0, 0, None, 0, None, 0, None, 0, 0, None, 0, None, 0, None, 0, None) == OK
    assert lib.dsnq_group_quant_bf16(0, 1536, A, 1536, 128, A, 1536, A, 0, 0, None) == OK
    assert lib.dsnq_group_quant_bf16(4, 1536, A, 1536, 32, A, 1536, A, 0, 0, None) == UNSUPPORTED
    assert lib.dsnq_quantize_weight_block128(0, 1536, A, 1536, A, 1536, A, 12, None) == OK
    assert lib.dsnq_quantize_weight_block128(4, 1500, A, 1500, A, 1536, A, 12, None) == UNSUPPORTED
    assert lib.dsnq_dual_rmsnorm_bf16(0, 1536, 512, A, 1536, A, 512, A, A, 1e-6, A, 1536, A, 512, None) == OK


def test_single_latent_argument_checks(lib):
    f = lib.dsnq_rmsnorm_group_quant
    assert f(0, 1536, None, 1536, None, 1e-6, 128, None, 1536, None, 0, 0, None) == OK     # empty call
    assert f(4, 1536, A, 1536, A, 1e-6, 64, A, 1536, A, 0, 0, None) == UNSUPPORTED        # group
    assert f(4, 1500, A, 1536, A, 1e-6, 128, A, 1536, A, 0, 0, None) == UNSUPPORTED       # K % 128
    assert f(4, 8192, A, 8192, A, 1e-6, 128, A, 8192, A, 0, 0, None) == UNSUPPORTED       # K > 4096
    assert f(4, 1536, A, 1000, A, 1e-6, 128, A, 1536, A, 0, 0, None) == INVALID           # ldx < K
    assert f(4, 1536, A, 1536, A, float("nan"), 128, A, 1536, A, 0, 0, None) == INVALID   # eps
    assert f(4, 1536, A + 8, 1536, A, 1e-6, 128, A, 1536, A, 0, 0, None) == MISALIGNED    # x
    assert f(4, 1536, A, 1540, A, 1e-6, 128, A, 1536, A, 0, 0, None) == MISALIGNED        # ldx
    assert f(4, 1536, A, 1536, A, 1e-6, 128, A, 1536, A, 1, 2, None) == INVALID           # col-major ld < M
    assert f(4, 1536, None, 1536, A, 1e-6, 128, A, 1536, A, 0, 0, None) == INVALID        # null x


def test_bf16_activation_gemm_argument_checks(lib):
    f = lib.dsnq_block_scaled_fp8_gemm_dual_bf16a

    def call(M=4, K=1536, a=A, lda=1536, N1=512, ldo1=512, N2=256, ws=(None, None)):
        return f(M, K, a, lda, N1, A, K, A, K // 128, A, ldo1, N2, A, K, A, K // 128, A, 256,
                 ws[0], ws[1], None)

    assert call(M=0) == OK
    assert call(M=-1) == INVALID
    assert call(K=1000, lda=1000) == UNSUPPORTED
    assert call(K=8192, lda=8192) == UNSUPPORTED           # K > 4096
    assert call(a=None) == INVALID
    assert call(N1=520, ldo1=520) == UNSUPPORTED           # N % 16
    assert call(N1=0, N2=0) == OK
    assert call(M=100) == INVALID                          # workspace needed above 64 rows
    assert call(M=100, ws=(A + 8, A)) == MISALIGNED
    assert call(lda=1000) == INVALID                       # in-kernel quant path (M <= 64)
    assert call(a=A + 8) == MISALIGNED
    assert call(lda=1540) == MISALIGNED


def test_python_and_library_agree_on_the_in_gemm_route(lib):
    """With a misaligned lda and no workspace, the in-GEMM route reports
    MISALIGNED and the two-launch route reports the missing workspace
    (INVALID): the library's dispatch is visible without a GPU."""
    import gemm_dsnq_dual_gb300 as dsnq
    f = lib.dsnq_block_scaled_fp8_gemm_dual_bf16a
    for K in range(128, 2048 + 256, 128):
        for M in range(1, 21):
            st = f(M, K, A, K + 4, 512, A, K, A, K // 128, A, 512, 0, None, 0, None, 0, None, 0, None, None, None)
            assert st in (MISALIGNED, INVALID), (M, K, st)
            assert (st == MISALIGNED) == dsnq.fused_quant_fits(M, K), (M, K)


def test_static_scratch_gemm_argument_checks(lib):
    f = lib.dsnq_block_scaled_fp8_gemm_dual_bf16a_static

    def call(M=4, K=1536):
        return f(M, K, A, K, 512, A, K, A, K // 128, A, 512, 256, A, K, A, K // 128, A, 256, None)

    assert call(M=0) == OK
    assert call(M=-1) == INVALID
    assert call(M=2049) == UNSUPPORTED                     # beyond the library's scratch
    assert call(K=2176) == UNSUPPORTED
    assert call(K=1000) == UNSUPPORTED                     # K % 128, fits the scratch
    # Same status as the workspace entry for the same bad input, whatever M is.
    g = lib.dsnq_block_scaled_fp8_gemm_dual_bf16a
    for M in (0, 4, 4096):
        st = f(M, 1536, A, 1536, -1, A, 1536, A, 12, A, 512, 256, A, 1536, A, 12, A, 256, None)
        assert st == INVALID, M
        assert g(M, 1536, A, 1536, -1, A, 1536, A, 12, A, 512, 256, A, 1536, A, 12, A, 256, None, None,
                 None) == INVALID, M


def test_fused_norm_quant_gemm_argument_checks(lib):
    f = lib.dsnq_fused_norm_quant_gemm_dual

    def call(M=4, Kq=1536, Kkv=512, q=A, ldq=2112, kv=A + 3072, ldkv=2112, eps=1e-6, kvo=A, N1=512, qf=None, qs=None):
        return f(M, Kq, Kkv, q, ldq, kv, ldkv, A, A, eps, kvo, Kkv, N1, A, Kq, A, Kq // 128, A, max(N1, 512),
                 256, A, Kq, A, Kq // 128, A, 256, qf, qs, None)

    assert call(M=0) == OK
    assert call(M=-1) == INVALID
    assert call(Kq=1000) == UNSUPPORTED
    assert call(Kkv=100) == UNSUPPORTED
    assert call(eps=float("nan")) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(q=None) == INVALID
    assert call(kvo=None) == INVALID
    assert call(ldq=1000) == INVALID
    assert call(q=A + 8) == MISALIGNED
    assert call(ldkv=2110) == MISALIGNED
    assert call(qf=A + 8, qs=A) == MISALIGNED
    assert call(N1=520) == UNSUPPORTED                     # N % 16
    assert call(M=100) == INVALID                          # q_fp8 / q_scale needed above a few rows


def test_gemm_plan_serves_every_k(lib):
    """Host-only plan of the GEMM: every M >= 1 and every K that is a
    multiple of 128 up to 8192 has a kernel variant whose shared memory fits
    one SM (227 KB); other K are refused before anything is launched."""
    v, b = C.c_int32(), C.c_int64()
    seen = set()
    for M in (1, 16, 17, 32, 33, 64, 65, 128, 255, 256, 300, 8192, 32768):
        for K in range(128, 8192 + 1, 128):
            assert lib.dsnq_gemm_plan(M, K, C.byref(v), C.byref(b)) == OK, (M, K)
            assert 0 < b.value <= 227 * 1024, (M, K, b.value)
            seen.add(v.value)
            if M <= 16:
                assert v.value == 1
            elif M <= 32:
                assert v.value == 2
            elif M <= 64:
                assert v.value == 3
            elif M < 256:
                assert v.value == (4 if K <= 4096 else 5), (M, K, v.value)
            else:
                assert v.value == (6 if K <= 4096 else 5), (M, K, v.value)
        assert lib.dsnq_gemm_plan(M, 8320, C.byref(v), C.byref(b)) == UNSUPPORTED
        assert lib.dsnq_gemm_plan(M, 1000, C.byref(v), C.byref(b)) == UNSUPPORTED
    assert seen == {1, 2, 3, 4, 5, 6}
    assert lib.dsnq_gemm_plan(0, 1536, C.byref(v), C.byref(b)) == OK and v.value == 0
    assert lib.dsnq_gemm_plan(-1, 1536, None, None) == INVALID
    # The calls themselves refuse K > 8192 on the host (no CUDA call is made here).
    assert gemm(lib, M=300, K=8320, lda=8320, ldw=8320, ldsw=65) == UNSUPPORTED


def test_bf16a_workspace_query(lib):
    c, s = C.c_int64(), C.c_int64()
    assert lib.dsnq_bf16a_workspace_bytes(1, 1536, C.byref(c), C.byref(s)) == OK
    assert (c.value, s.value) == (0, 0)                   # quantized inside the GEMM
    assert lib.dsnq_bf16a_workspace_bytes(100, 1536, C.byref(c), C.byref(s)) == OK
    assert (c.value, s.value) == (100 * 1536, 100 * 12 * 4)
    assert lib.dsnq_bf16a_workspace_bytes(0, 1536, C.byref(c), C.byref(s)) == OK
    assert (c.value, s.value) == (0, 0)
    assert lib.dsnq_bf16a_workspace_bytes(4, 8192, None, None) == UNSUPPORTED
    assert lib.dsnq_bf16a_workspace_bytes(-1, 1536, None, None) == INVALID


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "libdsnq.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _native.lib()
