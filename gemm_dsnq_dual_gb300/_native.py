"""ctypes loader for libdsnq.so (the C ABI declared in include/dsnq.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Loading fails loudly when the library has not been built; there is
no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
RELEASE_LIB_PATH = os.path.join(_PKG, "libdsnq.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libdsnq_debug.so")      # device index checks (DSNQ_DEBUG)
# DSNQ_DEBUG=1 in the environment selects the debug build.
LIB_PATH = DEBUG_LIB_PATH if os.environ.get("DSNQ_DEBUG") == "1" else RELEASE_LIB_PATH

DSNQ_OK = 0
STATUS_NAMES = {
    0: "DSNQ_OK", 1: "DSNQ_ERR_INVALID_ARG", 2: "DSNQ_ERR_MISALIGNED",
    3: "DSNQ_ERR_UNSUPPORTED", 4: "DSNQ_ERR_CUDA", 5: "DSNQ_ERR_TIMEOUT", 6: "DSNQ_ERR_BOUNDS",
}

i64, i32, u32, u64, f32, vp = C.c_int64, C.c_int32, C.c_uint32, C.c_uint64, C.c_float, C.c_void_p
pi64 = C.POINTER(C.c_int64)

# name -> (restype, argtypes); mirrors include/dsnq.h one to one.
SIGNATURES = {
    "dsnq_status_string": (C.c_char_p, [i32]),
    "dsnq_version": (i32, []),
    "dsnq_quant_output_sizes": (i32, [i64, i64, i32, i32, pi64, pi64]),
    "dsnq_fused_dual_rmsnorm_group_quant": (
        i32, [i64, i64, i64, vp, i64, vp, i64, vp, vp, f32, i32,
              vp, i64, vp, i32, i64, vp, i64, vp]),
    "dsnq_rmsnorm_group_quant": (i32, [i64, i64, vp, i64, vp, f32, i32, vp, i64, vp, i32, i64, vp]),
    "dsnq_dual_rmsnorm_bf16": (
        i32, [i64, i64, i64, vp, i64, vp, i64, vp, vp, f32, vp, i64, vp, i64, vp]),
    "dsnq_group_quant_bf16": (i32, [i64, i64, vp, i64, i32, vp, i64, vp, i32, i64, vp]),
    "dsnq_quantize_weight_block128": (i32, [i64, i64, vp, i64, vp, i64, vp, i64, vp]),
    "dsnq_block_scaled_fp8_gemm": (
        i32, [i64, i64, i64, vp, i64, vp, i32, i64, vp, i64, vp, i64, vp, i64, vp]),
    "dsnq_block_scaled_fp8_gemm_dual": (
        i32, [i64, i64, vp, i64, vp, i32, i64,
              i64, vp, i64, vp, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64, vp]),
    "dsnq_fused_norm_quant_gemm_dual": (
        i32, [i64, i64, i64, vp, i64, vp, i64, vp, vp, f32, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              vp, vp, vp]),
    "dsnq_block_scaled_fp8_gemm_dual_bf16a_static": (
        i32, [i64, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              vp]),
    "dsnq_block_scaled_fp8_gemm_dual_bf16a": (
        i32, [i64, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              i64, vp, i64, vp, i64, vp, i64,
              vp, vp, vp]),
    "dsnq_gemm_plan": (i32, [i64, i64, C.POINTER(C.c_int32), pi64]),
    "dsnq_bf16a_workspace_bytes": (i32, [i64, i64, pi64, pi64]),
    "dsnq_debug_status": (i32, [vp]),
    "dsnq_debug_build": (i32, []),
    "dsnq_debug_set": (None, [u32, u64]),
    "dsnq_set_launch_overlap": (None, [i32]),
}

_lib = None
_lock = threading.Lock()


class DsnqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {STATUS_NAMES.get(status, status)}")


def lib() -> C.CDLL:
    """The loaded library with argument types set."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is not built; run `python -m gemm_dsnq_dual_gb300.build`")
                h = C.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def use_library(path: str) -> None:
    """Load `path` (the release or the debug build) for every later call."""
    global _lib, LIB_PATH
    with _lock:
        LIB_PATH = path
        _lib = None


def check(status: int, where: str) -> None:
    if status != DSNQ_OK:
        raise DsnqError(status, where)
