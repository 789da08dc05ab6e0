"""GB300-native decode-step MLA latent pre-projection.

Thin PyTorch binding over libdsnq (include/dsnq.h).  Tensors supply device
memory and the current CUDA stream; every step runs in the library's CUDA
kernels.  Output tensors are allocated here with torch when not supplied.

  fused_dual_rmsnorm_group_quant  -- dual RMSNorm + per-1x128 FP8 quant (one kernel)
  block_scaled_fp8_gemm           -- W8A8 block-scaled GEMM on the pre-quantized pair
  block_scaled_fp8_gemm_dual      -- both wq_b consumers in one launch
  quantize_weight_block128        -- load-time 128x128 weight-block quantization
  dual_rmsnorm_bf16, group_quant_bf16 -- the unfused baseline sequence

Method: vLLM PR #53540 (fused_qk_rmsnorm_group_quant feeding
apply_pre_quantized_block_scaled_mm for the attention and indexer wq_b) and
sglang PR #27289 (transpose_scale: column-major activation scales).
"""

from __future__ import annotations

import ctypes as C

import torch

from ._native import DsnqError, check, lib  # noqa: F401

ROW_MAJOR = 0
COL_MAJOR = 1
GROUP = 128

__all__ = [
    "ROW_MAJOR", "COL_MAJOR", "DsnqError",
    "fused_dual_rmsnorm_group_quant", "rmsnorm_group_quant", "dual_rmsnorm_bf16", "group_quant_bf16",
    "quantize_weight_block128", "block_scaled_fp8_gemm", "block_scaled_fp8_gemm_dual",
    "block_scaled_fp8_gemm_dual_bf16a", "block_scaled_fp8_gemm_dual_bf16a_static", "fused_quant_fits",
    "bf16a_workspace_bytes", "gemm_plan",
    "fused_norm_quant_gemm_dual",
    "quant_output_sizes", "debug_status", "debug_set", "set_launch_overlap", "scale_layout_of", "scale_ld_for",
    "empty_scales",
]


def _stream(stream, dev) -> int:
    """The stream handle for a call on tensors of device `dev`.  The library
    launches on the current CUDA device (and picks per-device state by it), so
    tensors on another device are refused rather than silently mixed."""
    if dev.type != "cuda":
        raise ValueError(f"tensors must be CUDA tensors, got {dev}")
    cur = torch.cuda.current_device()
    if dev.index is not None and dev.index != cur:
        raise ValueError(f"tensors are on {dev} but the current CUDA device is cuda:{cur}; "
                         f"call under torch.cuda.device({dev})")
    if stream is None:
        stream = torch.cuda.current_stream(cur)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _layout(layout) -> int:
    if layout in (ROW_MAJOR, "row", "row_major"):
        return ROW_MAJOR
    if layout in (COL_MAJOR, "col", "col_major", "column_major"):
        return COL_MAJOR
    raise ValueError(f"unknown scale layout {layout!r}")


def _row_view_ok(t: torch.Tensor, name: str) -> int:
    """Row stride of a 2-D tensor whose rows are contiguous."""
    if t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError(f"{name} must be 2-D with contiguous rows")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def quant_output_sizes(M: int, Kq: int, group: int = GROUP, layout=ROW_MAJOR):
    """(n_scale_elems, default_ld_scale) of the scale buffer."""
    n, ld = C.c_int64(), C.c_int64()
    check(lib().dsnq_quant_output_sizes(M, Kq, group, _layout(layout), C.byref(n), C.byref(ld)),
          "dsnq_quant_output_sizes")
    return n.value, ld.value


def empty_scales(M: int, G: int, layout, device) -> torch.Tensor:
    """Logical [M, G] fp32 scale tensor in the requested memory layout
    (column-major = the transposed buffer viewed with strides (1, M))."""
    if _layout(layout) == ROW_MAJOR:
        return torch.empty(M, G, dtype=torch.float32, device=device)
    return torch.empty(G, M, dtype=torch.float32, device=device).t()


def scale_ld_for(scale: torch.Tensor, layout) -> int:
    """Leading dimension of a logical [M, G] scale tensor read in `layout`;
    raises if its memory does not have that layout."""
    M, G = scale.shape
    if _layout(layout) == ROW_MAJOR:
        if G > 1 and scale.stride(1) != 1:
            raise ValueError("scale tensor is not row-major")
        return scale.stride(0) if M > 1 else G
    if M > 1 and scale.stride(0) != 1:
        raise ValueError("scale tensor is not column-major")
    return scale.stride(1) if G > 1 else M


def scale_layout_of(scale: torch.Tensor):
    """(layout, ld) of a logical [M, G] scale tensor."""
    M, G = scale.shape
    if scale.stride(1) == 1 and (M <= 1 or scale.stride(0) >= G):
        return ROW_MAJOR, (scale.stride(0) if M > 1 else G)
    if scale.stride(0) == 1 and (G <= 1 or scale.stride(1) >= M):
        return COL_MAJOR, (scale.stride(1) if G > 1 else M)
    raise ValueError("scale tensor is neither row-major nor column-major")


def fused_dual_rmsnorm_group_quant(q, kv, gamma_q, gamma_kv, eps: float = 1e-6, group: int = GROUP,
                                   scale_layout=ROW_MAJOR, q_out=None, q_scale=None, kv_out=None,
                                   stream=None):
    """RMSNorm q [M,Kq] and kv [M,Kkv] (bf16, rows may be strided split views),
    quantize the normalized q per 1x128 group to E4M3FN.
    Returns (q_fp8 [M,Kq] float8_e4m3fn, q_scale [M,Kq/128] fp32, kv_out [M,Kkv] bf16)."""
    M, Kq = q.shape
    Kkv = kv.shape[1]
    dev = q.device
    lay = _layout(scale_layout)
    if q_out is None:
        q_out = torch.empty(M, Kq, dtype=torch.float8_e4m3fn, device=dev)
    if q_scale is None:
        q_scale = empty_scales(M, Kq // group, lay, dev)
    if kv_out is None:
        kv_out = torch.empty(M, Kkv, dtype=torch.bfloat16, device=dev)
    ld = scale_ld_for(q_scale, lay)
    check(lib().dsnq_fused_dual_rmsnorm_group_quant(
        M, Kq, Kkv, q.data_ptr(), _row_view_ok(q, "q"), kv.data_ptr(), _row_view_ok(kv, "kv"),
        gamma_q.data_ptr(), gamma_kv.data_ptr(), float(eps), group,
        q_out.data_ptr(), _row_view_ok(q_out, "q_out"), q_scale.data_ptr(), lay, ld,
        kv_out.data_ptr(), _row_view_ok(kv_out, "kv_out"), _stream(stream, q.device)),
        "dsnq_fused_dual_rmsnorm_group_quant")
    return q_out, q_scale, kv_out


def rmsnorm_group_quant(x, gamma, eps: float = 1e-6, group: int = GROUP, scale_layout=ROW_MAJOR,
                        x_out=None, x_scale=None, stream=None):
    """RMSNorm one latent x [M,K] (bf16, rows may be a strided view) and
    quantize it per 1x128 group to E4M3FN.  Returns (x_fp8, x_scale)."""
    M, K = x.shape
    lay = _layout(scale_layout)
    if x_out is None:
        x_out = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=x.device)
    if x_scale is None:
        x_scale = empty_scales(M, K // group, lay, x.device)
    ld = scale_ld_for(x_scale, lay)
    check(lib().dsnq_rmsnorm_group_quant(
        M, K, x.data_ptr(), _row_view_ok(x, "x"), gamma.data_ptr(), float(eps), group,
        x_out.data_ptr(), _row_view_ok(x_out, "x_out"), x_scale.data_ptr(), lay, ld, _stream(stream, x.device)),
        "dsnq_rmsnorm_group_quant")
    return x_out, x_scale


def dual_rmsnorm_bf16(q, kv, gamma_q, gamma_kv, eps: float = 1e-6, q_out=None, kv_out=None, stream=None):
    """Unfused baseline step 1: both latents normalized to bf16."""
    M, Kq = q.shape
    Kkv = kv.shape[1]
    if q_out is None:
        q_out = torch.empty(M, Kq, dtype=torch.bfloat16, device=q.device)
    if kv_out is None:
        kv_out = torch.empty(M, Kkv, dtype=torch.bfloat16, device=q.device)
    check(lib().dsnq_dual_rmsnorm_bf16(
        M, Kq, Kkv, q.data_ptr(), _row_view_ok(q, "q"), kv.data_ptr(), _row_view_ok(kv, "kv"),
        gamma_q.data_ptr(), gamma_kv.data_ptr(), float(eps),
        q_out.data_ptr(), _row_view_ok(q_out, "q_out"), kv_out.data_ptr(), _row_view_ok(kv_out, "kv_out"),
        _stream(stream, q.device)), "dsnq_dual_rmsnorm_bf16")
    return q_out, kv_out


def group_quant_bf16(x, group: int = GROUP, scale_layout=ROW_MAJOR, x_out=None, x_scale=None, stream=None):
    """Unfused baseline step 2: per-1x128 quant of a bf16 [M,K] tensor."""
    M, K = x.shape
    lay = _layout(scale_layout)
    if x_out is None:
        x_out = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=x.device)
    if x_scale is None:
        x_scale = empty_scales(M, K // group, lay, x.device)
    ld = scale_ld_for(x_scale, lay)
    check(lib().dsnq_group_quant_bf16(
        M, K, x.data_ptr(), _row_view_ok(x, "x"), group, x_out.data_ptr(), _row_view_ok(x_out, "x_out"),
        x_scale.data_ptr(), lay, ld, _stream(stream, x.device)), "dsnq_group_quant_bf16")
    return x_out, x_scale


def quantize_weight_block128(w, w_out=None, w_scale=None, stream=None):
    """fp32 weight [N,K] -> (E4M3FN codes [N,K], fp32 block scales [ceil(N/128), K/128])."""
    N, K = w.shape
    if w_out is None:
        w_out = torch.empty(N, K, dtype=torch.float8_e4m3fn, device=w.device)
    if w_scale is None:
        w_scale = torch.empty((N + 127) // 128, K // 128, dtype=torch.float32, device=w.device)
    check(lib().dsnq_quantize_weight_block128(
        N, K, w.data_ptr(), _row_view_ok(w, "w"), w_out.data_ptr(), _row_view_ok(w_out, "w_out"),
        w_scale.data_ptr(), _row_view_ok(w_scale, "w_scale"), _stream(stream, w.device)),
        "dsnq_quantize_weight_block128")
    return w_out, w_scale


def block_scaled_fp8_gemm(a_fp8, a_scale, w_fp8, w_scale, out=None, stream=None):
    """out[M,N] bf16 = block-scaled (a_fp8, a_scale) x (w_fp8, w_scale)^T."""
    M, K = a_fp8.shape
    N = w_fp8.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=a_fp8.device)
    lay, ld = scale_layout_of(a_scale)
    check(lib().dsnq_block_scaled_fp8_gemm(
        M, N, K, a_fp8.data_ptr(), _row_view_ok(a_fp8, "a_fp8"), a_scale.data_ptr(), lay, ld,
        w_fp8.data_ptr(), _row_view_ok(w_fp8, "w_fp8"), w_scale.data_ptr(), _row_view_ok(w_scale, "w_scale"),
        out.data_ptr(), _row_view_ok(out, "out"), _stream(stream, a_fp8.device)), "dsnq_block_scaled_fp8_gemm")
    return out


def block_scaled_fp8_gemm_dual(a_fp8, a_scale, w1_fp8, w1_scale, w2_fp8, w2_scale,
                               out1=None, out2=None, stream=None):
    """Both consumers (e.g. attention wq_b and indexer wq_b) in one launch."""
    M, K = a_fp8.shape
    N1, N2 = w1_fp8.shape[0], w2_fp8.shape[0]
    dev = a_fp8.device
    if out1 is None:
        out1 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    if out2 is None:
        out2 = torch.empty(M, N2, dtype=torch.bfloat16, device=dev)
    lay, ld = scale_layout_of(a_scale)
    check(lib().dsnq_block_scaled_fp8_gemm_dual(
        M, K, a_fp8.data_ptr(), _row_view_ok(a_fp8, "a_fp8"), a_scale.data_ptr(), lay, ld,
        N1, w1_fp8.data_ptr(), _row_view_ok(w1_fp8, "w1_fp8"), w1_scale.data_ptr(),
        _row_view_ok(w1_scale, "w1_scale"), out1.data_ptr(), _row_view_ok(out1, "out1"),
        N2, w2_fp8.data_ptr(), _row_view_ok(w2_fp8, "w2_fp8"), w2_scale.data_ptr(),
        _row_view_ok(w2_scale, "w2_scale"), out2.data_ptr(), _row_view_ok(out2, "out2"),
        _stream(stream, a_fp8.device)), "dsnq_block_scaled_fp8_gemm_dual")
    return out1, out2


def bf16a_workspace_bytes(M: int, K: int):
    """(code_bytes, scale_bytes) of the workspace block_scaled_fp8_gemm_dual_bf16a
    needs for M rows of K bf16 activations; (0, 0) when it quantizes inside
    the GEMM (the library's own rule, dsnq_bf16a_workspace_bytes)."""
    c, s = C.c_int64(), C.c_int64()
    check(lib().dsnq_bf16a_workspace_bytes(M, K, C.byref(c), C.byref(s)), "dsnq_bf16a_workspace_bytes")
    return c.value, s.value


def fused_quant_fits(M: int, K: int) -> bool:
    """True when block_scaled_fp8_gemm_dual_bf16a quantizes inside the GEMM
    (one launch, no workspace)."""
    return M > 0 and bf16a_workspace_bytes(M, K) == (0, 0)


def gemm_plan(M: int, K: int):
    """(variant, dynamic shared memory bytes) of the GEMM kernel that
    block_scaled_fp8_gemm(_dual) launches for M rows and reduction length K
    (host-only query, dsnq_gemm_plan)."""
    v, b = C.c_int32(), C.c_int64()
    check(lib().dsnq_gemm_plan(M, K, C.byref(v), C.byref(b)), "dsnq_gemm_plan")
    return v.value, b.value


def block_scaled_fp8_gemm_dual_bf16a(a_bf16, w1_fp8, w1_scale, w2_fp8, w2_scale,
                                     out1=None, out2=None, workspace=None, stream=None):
    """The dual GEMM on bf16 activations, quantized per 1x128 on the fly.
    `workspace` = (a_fp8 [M,K] uint8/e4m3, a_scale [M*K/128] fp32) is only
    needed outside fused_quant_fits(M, K); it is allocated here if omitted."""
    M, K = a_bf16.shape
    N1, N2 = w1_fp8.shape[0], w2_fp8.shape[0]
    dev = a_bf16.device
    if out1 is None:
        out1 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    if out2 is None:
        out2 = torch.empty(M, N2, dtype=torch.bfloat16, device=dev)
    ws_a = ws_s = 0
    code_bytes, scale_bytes = bf16a_workspace_bytes(M, K)
    if code_bytes:
        if workspace is None:
            workspace = (torch.empty(code_bytes, dtype=torch.uint8, device=dev),
                         torch.empty(scale_bytes // 4, dtype=torch.float32, device=dev))
        ws_a, ws_s = workspace[0].data_ptr(), workspace[1].data_ptr()
    check(lib().dsnq_block_scaled_fp8_gemm_dual_bf16a(
        M, K, a_bf16.data_ptr(), _row_view_ok(a_bf16, "a_bf16"),
        N1, w1_fp8.data_ptr(), _row_view_ok(w1_fp8, "w1_fp8"), w1_scale.data_ptr(),
        _row_view_ok(w1_scale, "w1_scale"), out1.data_ptr(), _row_view_ok(out1, "out1"),
        N2, w2_fp8.data_ptr(), _row_view_ok(w2_fp8, "w2_fp8"), w2_scale.data_ptr(),
        _row_view_ok(w2_scale, "w2_scale"), out2.data_ptr(), _row_view_ok(out2, "out2"),
        ws_a, ws_s, _stream(stream, a_bf16.device)), "dsnq_block_scaled_fp8_gemm_dual_bf16a")
    return out1, out2


def block_scaled_fp8_gemm_dual_bf16a_static(a_bf16, w1_fp8, w1_scale, w2_fp8, w2_scale,
                                            out1=None, out2=None, stream=None):
    """block_scaled_fp8_gemm_dual_bf16a with the library's own device scratch
    (M, K <= 2048): nothing is allocated for the quantized pair."""
    M, K = a_bf16.shape
    N1, N2 = w1_fp8.shape[0], w2_fp8.shape[0]
    dev = a_bf16.device
    if out1 is None:
        out1 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    if out2 is None:
        out2 = torch.empty(M, N2, dtype=torch.bfloat16, device=dev)
    check(lib().dsnq_block_scaled_fp8_gemm_dual_bf16a_static(
        M, K, a_bf16.data_ptr(), _row_view_ok(a_bf16, "a_bf16"),
        N1, w1_fp8.data_ptr(), _row_view_ok(w1_fp8, "w1_fp8"), w1_scale.data_ptr(),
        _row_view_ok(w1_scale, "w1_scale"), out1.data_ptr(), _row_view_ok(out1, "out1"),
        N2, w2_fp8.data_ptr(), _row_view_ok(w2_fp8, "w2_fp8"), w2_scale.data_ptr(),
        _row_view_ok(w2_scale, "w2_scale"), out2.data_ptr(), _row_view_ok(out2, "out2"),
        _stream(stream, a_bf16.device)), "dsnq_block_scaled_fp8_gemm_dual_bf16a_static")
    return out1, out2


def fused_norm_quant_gemm_dual(q, kv, gamma_q, gamma_kv, eps, w1_fp8, w1_scale, w2_fp8, w2_scale,
                               out1=None, out2=None, kv_out=None, q_fp8=None, q_scale=None, stream=None):
    """RMSNorm + per-1x128 quant of the q latent (kv latent normalized to
    bf16), then the dual GEMM, in one call.  Returns (out1, out2, kv_out,
    q_fp8, q_scale); the last two are None when the rows were quantized
    inside the GEMM and no buffers were passed."""
    M, Kq = q.shape
    Kkv = kv.shape[1]
    N1, N2 = w1_fp8.shape[0], w2_fp8.shape[0]
    dev = q.device
    if out1 is None:
        out1 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    if out2 is None:
        out2 = torch.empty(M, N2, dtype=torch.bfloat16, device=dev)
    if kv_out is None:
        kv_out = torch.empty(M, Kkv, dtype=torch.bfloat16, device=dev)
    one_launch = fused_quant_fits(M, Kq) and Kkv <= 2048 and N1 + N2 > 0
    if not one_launch and M > 0:
        if q_fp8 is None:
            q_fp8 = torch.empty(M, Kq, dtype=torch.float8_e4m3fn, device=dev)
        if q_scale is None:
            q_scale = empty_scales(M, Kq // GROUP, COL_MAJOR, dev)
    if q_fp8 is not None and not q_fp8.is_contiguous():
        raise ValueError("q_fp8 must be contiguous [M, Kq]")
    if q_scale is not None and M > 1 and q_scale.stride() != (1, M):
        raise ValueError("q_scale must be column-major [M, Kq/128] (strides (1, M))")
    check(lib().dsnq_fused_norm_quant_gemm_dual(
        M, Kq, Kkv, q.data_ptr(), _row_view_ok(q, "q"), kv.data_ptr(), _row_view_ok(kv, "kv"),
        gamma_q.data_ptr(), gamma_kv.data_ptr(), float(eps), kv_out.data_ptr(), _row_view_ok(kv_out, "kv_out"),
        N1, w1_fp8.data_ptr(), _row_view_ok(w1_fp8, "w1_fp8"), w1_scale.data_ptr(),
        _row_view_ok(w1_scale, "w1_scale"), out1.data_ptr(), _row_view_ok(out1, "out1"),
        N2, w2_fp8.data_ptr(), _row_view_ok(w2_fp8, "w2_fp8"), w2_scale.data_ptr(),
        _row_view_ok(w2_scale, "w2_scale"), out2.data_ptr(), _row_view_ok(out2, "out2"),
        0 if q_fp8 is None else q_fp8.data_ptr(), 0 if q_scale is None else q_scale.data_ptr(),
        _stream(stream, q.device)), "dsnq_fused_norm_quant_gemm_dual")
    return out1, out2, kv_out, q_fp8, q_scale


def debug_status(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device status."""
    return lib().dsnq_debug_status(_stream(stream, torch.device("cuda", torch.cuda.current_device())))


def debug_set(inject_flags: int = 0, wait_timeout_ns: int = 0) -> None:
    lib().dsnq_debug_set(inject_flags, wait_timeout_ns)


def set_launch_overlap(enable: bool = True) -> None:
    """Programmatic dependent launch for every later call (on by default):
    a kernel may be scheduled while the previous kernel of its stream runs,
    and waits in hardware for that kernel's writes before reading inputs."""
    lib().dsnq_set_launch_overlap(1 if enable else 0)
