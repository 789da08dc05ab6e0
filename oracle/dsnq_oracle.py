"""fp64 CPU oracle for the decode-step MLA latent pre-projection.

TEST INFRASTRUCTURE ONLY.  This module is the independent definition that the
CUDA path is checked against.  Only the test suite, the package's smoke check
and the benchmark's CPU-baseline leg may import it; the product path never
does, and this module imports nothing from the product package.

What it computes (the method of vLLM PR #53540, "[ROCm] fused DSv4 q/kv
RMSNorm + q FP8 per-1x128 group quant", and of sglang PR #27289,
"transpose_scale"):

  1. Dual RMSNorm of the q-lora latent (width Kq) and the kv latent (width
     Kkv) of each token row, accumulated wider than the bf16 inputs
     (PR #53540 body, "Purpose": both latents are RMSNormed with fp32
     accumulation).  Here everything is fp64.
  2. Per-1x128 dynamic group quantization of the normalized q latent to FP8
     E4M3FN with fp32 scales, taken from the fp32 normalized values, not from
     a bf16 copy (PR #53540 body, "Purpose": quantization reads the fp32
     accumulator, single rounding).
  3. The normalized kv latent rounded to bf16 (PR #53540 prhub summary,
     custom-op snippet: kv_normed has kv's dtype).
  4. The scales written row-major [M, Kq/128] or column-major, element
     (m, g) at g*ld + m (sglang PR #27289, fp8_utils snippet: the transposed
     scale is the same logical shape with strides (1, M)).
  5. The W8A8 block-scaled GEMM that consumes the pre-quantized pair:
     out[m, n] = sum_k dec(a[m,k]) * sa[m, k/128] * dec(w[n,k]) * sw[n/128, k/128]
     (PR #53540 prhub summary, rocm.py snippet
     apply_pre_quantized_block_scaled_mm(A=x_fp8, B=weight, As=x_scale,
     Bs=weight_scale); sglang PR #27289, aiter_w8a8_block_fp8_linear with
     block_size [128, 128]).

Readings where the pages are silent (each is also listed in the design notes):
  * RMSNorm is x / sqrt(mean(x^2) + eps) * gamma, eps inside the root, one
    eps for both latents (the shared-path snippet passes self.eps to both).
  * The scale is amax / 448 (448 = largest finite E4M3FN value) in fp32; an
    all-zero group gets scale 0 and zero codes (sign kept).
  * The quantize step works on fp32 operands, as the pages place it ("reads
    the fp32 accumulator"): the normalized value is rounded to fp32 and the
    quotient x / scale is one IEEE fp32 division before the E4M3 rounding.
  * E4M3FN encoding rounds to nearest, ties to even, and saturates to +-448.
  * The weight-scale tensor (weight_scale or weight_scale_inv) multiplies.

Every function here is parity-pinned by tests that do not re-use its own
formulas: exhaustive codec round trips, library special cases
(torch float8_e4m3fn / bfloat16 casts, torch rms_norm and matmul in float64),
closed forms, hand-computed cases and invariants.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0          # largest finite E4M3FN magnitude, code 0x7E
E4M3_MIN_NORMAL_EXP = -6  # smallest normal exponent; subnormal spacing 2**-9
GROUP = 128               # per-1x128 activation groups, 128x128 weight blocks

SCALE_ROW_MAJOR = 0
SCALE_COL_MAJOR = 1


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16): the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _round_to_grid(a: np.ndarray, frac_bits: int, min_exp: int) -> np.ndarray:
    """Round non-negative fp64 magnitudes to a binary format with `frac_bits`
    stored fraction bits and smallest normal exponent `min_exp`, ties to even.

    The grid spacing in the binade [2**e, 2**(e+1)) is 2**(e - frac_bits);
    below 2**min_exp the subnormal spacing 2**(min_exp - frac_bits) applies.
    Division by a power of two and np.rint are exact, so the only rounding is
    the ties-to-even one of np.rint."""
    _, ex = np.frexp(a)               # a = f * 2**ex, 0.5 <= f < 1
    e = np.maximum(ex - 1, min_exp)   # binade exponent, clamped at subnormals
    quantum = np.ldexp(1.0, e - frac_bits)
    return np.rint(a / quantum) * quantum


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 round-to-nearest-even of fp64 values, as uint16 bit patterns
    (one rounding straight from fp64, no fp32 intermediate)."""
    x = np.asarray(x, dtype=np.float64)
    r = _round_to_grid(np.abs(x), 7, -126)
    r = np.where(np.signbit(x), -r, r)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3FN code (uint8) of fp64 values: bias 7, no infinities,
    round to nearest with ties to even, saturating to +-448.  The sign bit is
    copied from the input, so negative values that round to zero give 0x80."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    v = np.minimum(_round_to_grid(a, 3, E4M3_MIN_NORMAL_EXP), E4M3_MAX)
    # Bit pattern of the rounded magnitude v.
    _, ex = np.frexp(v)
    e = ex - 1
    normal = v >= 2.0 ** E4M3_MIN_NORMAL_EXP
    sub_code = np.rint(v / 2.0 ** -9)                     # 0..7 below 2**-6
    e_n = np.where(normal, e, 0)
    frac = np.where(normal, v / np.ldexp(1.0, e_n) - 1.0, 0.0)
    norm_code = (e_n + 7) * 8 + np.rint(frac * 8.0)
    code = np.where(normal, norm_code, sub_code).astype(np.int64)
    code = code | np.where(np.signbit(x), 0x80, 0)
    return code.astype(np.uint8)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """Value of E4M3FN codes (NaN for S.1111.111)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(E == 0, m * 2.0 ** -9,
                   (1.0 + m / 8.0) * np.ldexp(1.0, E - 7))
    mag = np.where((E == 15) & (m == 7), np.nan, mag)
    return sign * mag


# ---------------------------------------------------------------------------
# Fused dual RMSNorm + per-1x128 group quant (the first kernel of the path)
# ---------------------------------------------------------------------------

def rmsnorm_f64(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise x / sqrt(mean(x^2) + eps) * gamma in fp64."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.sum(x * x, axis=-1, keepdims=True) / x.shape[-1]
    r = 1.0 / np.sqrt(ms + np.float64(eps))
    return x * r * np.asarray(gamma, dtype=np.float64)


def group_quant_f64(xhat: np.ndarray, group: int = GROUP):
    """Per-1x`group` quantization to E4M3FN of values that the method holds
    in fp32 (the normalized latent "read from the fp32 accumulator", PR #53540
    "Purpose"; a bf16 tensor; an fp32 weight).

    Returns (codes uint8 [M, K], scales float32 [M, K/group] logical).
    The quantize step is taken in fp32, the precision the pages give it:
      x32   = fp32(x)                      (exact for bf16 and fp32 inputs)
      scale = fp32(max|x32| / 448)
      code  = e4m3(fp32(x32 / scale))      (IEEE fp32 divide, then RNE to E4M3)
    A group whose scale is 0 gets the quotient x * 0 (signed zero)."""
    x32 = np.asarray(xhat, dtype=np.float64).astype(np.float32)
    M, K = x32.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    g = x32.reshape(M, K // group, group)
    amax = np.max(np.abs(g), axis=-1)
    scale = amax / np.float32(E4M3_MAX)              # fp32 / fp32: one IEEE rounding
    s = scale[..., None]
    safe = np.where(s > 0, s, np.float32(1.0))
    quot = np.where(s > 0, g / safe, g * np.float32(0.0))   # fp32 quotient
    codes = e4m3_encode(quot.astype(np.float64)).reshape(M, K)
    return codes, scale.astype(np.float32)


def store_scales(scale: np.ndarray, layout: int, ld: int | None = None) -> np.ndarray:
    """Lay the logical [M, G] fp32 scales out in memory.

    Row-major: element (m, g) at m*ld + g (ld >= G, default G).
    Column-major: element (m, g) at g*ld + m (ld >= M, default M), i.e. the
    transposed copy viewed with strides (1, ld).  Unwritten slots stay NaN."""
    M, G = scale.shape
    if layout == SCALE_ROW_MAJOR:
        ld = G if ld is None else ld
        buf = np.full(max(M - 1, 0) * ld + G if M else 0, np.nan, dtype=np.float32)
        for m in range(M):
            buf[m * ld:m * ld + G] = scale[m]
    elif layout == SCALE_COL_MAJOR:
        ld = M if ld is None else ld
        buf = np.full(max(G - 1, 0) * ld + M if M else 0, np.nan, dtype=np.float32)
        for g in range(G):
            buf[g * ld:g * ld + M] = scale[:, g]
    else:
        raise ValueError("unknown scale layout")
    return buf


def load_scales(buf: np.ndarray, M: int, G: int, layout: int, ld: int | None = None) -> np.ndarray:
    """Inverse of store_scales: the logical [M, G] view of a scale buffer."""
    buf = np.asarray(buf, dtype=np.float32)
    out = np.empty((M, G), dtype=np.float32)
    if layout == SCALE_ROW_MAJOR:
        ld = G if ld is None else ld
        for m in range(M):
            out[m] = buf[m * ld:m * ld + G]
    else:
        ld = M if ld is None else ld
        for g in range(G):
            out[:, g] = buf[g * ld:g * ld + M]
    return out


def fused_dual_rmsnorm_group_quant(q_bits, kv_bits, gamma_q_bits, gamma_kv_bits,
                                   eps: float, group: int = GROUP):
    """The fused op: returns (q_codes uint8 [M,Kq], q_scale float32 [M,Kq/group]
    logical, kv_out bf16 bits uint16 [M,Kkv]).

    Inputs are bf16 bit patterns (uint16); eps is taken at its fp32 value,
    the precision in which the library's API receives it."""
    eps = float(np.float32(eps))
    q = bf16_bits_to_f64(q_bits)
    kv = bf16_bits_to_f64(kv_bits)
    xq = rmsnorm_f64(q, bf16_bits_to_f64(gamma_q_bits), eps)
    xkv = rmsnorm_f64(kv, bf16_bits_to_f64(gamma_kv_bits), eps)
    codes, scale = group_quant_f64(xq, group)
    return codes, scale, f64_to_bf16_bits(xkv)


def rmsnorm_group_quant(x_bits, gamma_bits, eps: float, group: int = GROUP):
    """Single-latent RMSNorm + per-1x128 group quant (sglang PR #27289,
    fused_rms_fp8_group_quant): the q part of the fused op for one latent.
    Returns (codes uint8 [M,K], scale float32 [M,K/group] logical)."""
    eps = float(np.float32(eps))
    x = rmsnorm_f64(bf16_bits_to_f64(x_bits), bf16_bits_to_f64(gamma_bits), eps)
    return group_quant_f64(x, group)


def normalized_latents(q_bits, kv_bits, gamma_q_bits, gamma_kv_bits, eps: float):
    """The unrounded fp64 normalized latents (x_hat_q, x_hat_kv)."""
    eps = float(np.float32(eps))
    return (rmsnorm_f64(bf16_bits_to_f64(q_bits), bf16_bits_to_f64(gamma_q_bits), eps),
            rmsnorm_f64(bf16_bits_to_f64(kv_bits), bf16_bits_to_f64(gamma_kv_bits), eps))


# ---------------------------------------------------------------------------
# The unfused sequence the fusion replaces (shared path of PR #53540:
# fused_q_kv_rmsnorm to bf16, then per-1x128 quant of the bf16 q, twice)
# ---------------------------------------------------------------------------

def dual_rmsnorm_bf16(q_bits, kv_bits, gamma_q_bits, gamma_kv_bits, eps: float):
    """Baseline step 1: both latents normalized and rounded to bf16 bits."""
    xq, xkv = normalized_latents(q_bits, kv_bits, gamma_q_bits, gamma_kv_bits, eps)
    return f64_to_bf16_bits(xq), f64_to_bf16_bits(xkv)


def group_quant_bf16(x_bits, group: int = GROUP):
    """Baseline step 2: per-1x128 quant of a bf16 tensor (its exact values)."""
    return group_quant_f64(bf16_bits_to_f64(x_bits), group)


# ---------------------------------------------------------------------------
# Weights and the block-scaled GEMM (the second kernel of the path)
# ---------------------------------------------------------------------------

def quantize_weight_block128(w: np.ndarray):
    """Per-128x128-block quantization of a weight [N, K] (fp32 values) to
    E4M3FN codes with fp32 block scales [ceil(N/128), K/128].  Same rule as the
    activation groups, in fp32: scale = fp32(amax/448),
    code = e4m3(fp32(w / scale))."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    nb, kb = -(-N // GROUP), K // GROUP
    codes = np.empty((N, K), dtype=np.uint8)
    scale = np.empty((nb, kb), dtype=np.float32)
    for i in range(nb):
        rows = slice(i * GROUP, min(N, (i + 1) * GROUP))
        for j in range(kb):
            cols = slice(j * GROUP, (j + 1) * GROUP)
            blk = w[rows, cols]
            s = np.max(np.abs(blk)) / np.float32(E4M3_MAX)
            scale[i, j] = s
            quot = blk / s if s > 0 else blk * np.float32(0.0)
            codes[rows, cols] = e4m3_encode(quot.astype(np.float64))
    return codes, scale


def dequantize_activation(a_codes: np.ndarray, a_scale: np.ndarray) -> np.ndarray:
    """dec(a[m,k]) * sa[m, k/128] in fp64; a_scale is the logical [M, K/128]."""
    sa = np.repeat(np.asarray(a_scale, dtype=np.float64), GROUP, axis=1)
    return e4m3_decode(a_codes) * sa


def dequantize_weight(w_codes: np.ndarray, w_scale: np.ndarray) -> np.ndarray:
    """dec(w[n,k]) * sw[n/128, k/128] in fp64."""
    N, _ = w_codes.shape
    sw = np.repeat(np.repeat(np.asarray(w_scale, dtype=np.float64), GROUP, axis=0)[:N],
                   GROUP, axis=1)
    return e4m3_decode(w_codes) * sw


def block_scaled_gemm(a_codes, a_scale, w_codes, w_scale, rows=None) -> np.ndarray:
    """out[m, n] = sum_k dec(a[m,k]) sa[m,k/128] dec(w[n,k]) sw[n/128,k/128],
    fp64, for the rows `rows` of A (all rows by default).  The dequantize-then-
    multiply order equals the per-K-block promotion of the definition exactly
    in real arithmetic."""
    a_codes = np.asarray(a_codes)
    a_scale = np.asarray(a_scale)
    if rows is not None:
        a_codes, a_scale = a_codes[rows], a_scale[rows]
    return dequantize_activation(a_codes, a_scale) @ dequantize_weight(w_codes, w_scale).T


def output_bf16_bits(out_f64: np.ndarray) -> np.ndarray:
    """The bf16 rounding of the GEMM output."""
    return f64_to_bf16_bits(out_f64)
