// Per-1x128 FP8 group quantization arithmetic shared by the norm+quant
// kernels and the GEMM that quantizes its bf16 activations itself, so that
// both take every quantization decision identically.
//
// Definition (vLLM PR #53540 "Purpose"; sglang PR #27289, per-1x128 quant):
// for a group of 128 fp32 values x with amax = max |x|,
//   scale = fp32(amax / 448)                       (IEEE division, one rounding)
//   code  = e4m3_rn_satfinite(fp32(x / scale))     (0 codes, signed, when amax = 0)
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace dsnq {

constexpr float kE4M3Max = 448.0f;  // largest finite E4M3FN value

// ---- packed fp32 pairs: the f32x2 arithmetic of sm_100+ through the CUDA
// builtins (one instruction per pair).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Eight bf16 of a 16-byte chunk as four fp32 pairs (exact: bf16 is the top
// half of an fp32).
__device__ __forceinline__ void unpack8(const uint4& v, float2 (&f)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t e4m3x2(float2 v) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Sum over the 32 lanes (butterfly: every lane gets the same value).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct GroupQuant {
    float scale;            // amax / 448, IEEE fp32
    float2 ylo, yhi;        // fp32(1/scale) * (1 -+ 2^-20), rounded: bracket the quotient
    bool exact;             // reciprocal not finite: divide
};

// scale = RN(amax / 448) by the correction step of Markstein's division
// method: with y = RN(1/448), q0 = RN(amax * y) and the exact remainder
// amax - q0 * 448 (one FMA), RN(q0 + remainder * y) is the correctly rounded
// quotient for every amax >= 2^-96 (checked exhaustively over a binade, and
// across binades, in the test suite); below that, the division.
__device__ __forceinline__ float group_scale(float amax) {
    constexpr float kRecip448 = 1.0f / kE4M3Max;
    const float q0 = __fmul_rn(amax, kRecip448);
    float scale = fmaf(fmaf(-q0, kE4M3Max, amax), kRecip448, q0);
    if (amax < 0x1p-96f) scale = amax / kE4M3Max;
    return scale;
}

// Groups whose scale is too small for a finite reciprocal take the division.
__device__ __forceinline__ bool group_needs_division(float scale) { return scale > 0.f && scale < 1.0e-36f; }

// The reciprocal the bracket scales (0 for an all-zero group and for groups
// that take the division): within 2^-22 of 1/scale (fast divide, 2 ulp).
__device__ __forceinline__ float group_recip(float scale) {
    return (scale > 0.f && !group_needs_division(scale)) ? __fdividef(1.0f, scale) : 0.f;
}

// The bracket of a group from its scale and reciprocal.  Each product below
// adds at most 2^-24 to the reciprocal's 2^-22, so x*ylo <= x/scale <= x*yhi
// (in magnitude order) with room to spare.
__device__ __forceinline__ GroupQuant group_quant_from(float scale, float y) {
    GroupQuant gq;
    gq.scale = scale;
    gq.exact = group_needs_division(scale);
    const float lo = y * (1.0f - 0x1p-20f), hi = y * (1.0f + 0x1p-20f);
    gq.ylo = make_float2(lo, lo);
    gq.yhi = make_float2(hi, hi);
    return gq;
}

__device__ __forceinline__ GroupQuant make_group_quant(float amax) {
    const float scale = group_scale(amax);
    return group_quant_from(scale, group_recip(scale));
}

// Codes of eight values by the bracket (E4M3 rounding is monotone, so when
// both ends of the bracket give the same code, that is the code of the exact
// quotient); *ok is false when a code is not determined (the quotient lies
// within 2^-20 of a rounding boundary) or the group needs the division.
__device__ __forceinline__ uint2 quant8_bracket(const float2 (&f)[4], const GroupQuant& gq, bool& ok) {
    uint32_t lo[2], hi[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        lo[w] = e4m3x2(mul2(f[2 * w], gq.ylo)) | (e4m3x2(mul2(f[2 * w + 1], gq.ylo)) << 16);
        hi[w] = e4m3x2(mul2(f[2 * w], gq.yhi)) | (e4m3x2(mul2(f[2 * w + 1], gq.yhi)) << 16);
    }
    ok = lo[0] == hi[0] && lo[1] == hi[1] && !gq.exact;
    return make_uint2(lo[0], lo[1]);
}

// Codes of eight values by the IEEE division itself (the rare undetermined
// case, and all-zero groups: signed zero codes).
__device__ __forceinline__ uint2 quant8_divide(const float2 (&f)[4], float scale) {
    float2 qv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        qv[i] = scale > 0.f ? make_float2(__fdiv_rn(f[i].x, scale), __fdiv_rn(f[i].y, scale))
                            : make_float2(f[i].x * 0.f, f[i].y * 0.f);
    return make_uint2(e4m3x2(qv[0]) | (e4m3x2(qv[1]) << 16), e4m3x2(qv[2]) | (e4m3x2(qv[3]) << 16));
}

}  // namespace dsnq
