// Fused dual RMSNorm + per-1x128 FP8 group quant, the two unfused baseline
// kernels it replaces, and the load-time 128x128 weight-block quantizer.
//
// Method: vLLM PR #53540 ("Purpose"): RMSNorm both MLA latents with fp32
// accumulation and quantize the normalized q latent per 1x128 group to FP8
// with fp32 scales in the same pass, reading the fp32 values (one rounding);
// kv stays bf16.  Scale layout switch: sglang PR #27289 ("transpose_scale").
//
// Kernel shape (one CTA = one warp-group; rows are processed in a
// grid-stride loop so the per-thread set-up is paid once per CTA):
//   * a row is cut into 16-byte chunks of 8 bf16; chunk c < Kq/8 is q, the
//     rest is kv.  Thread t owns chunks t, t+128, ... (PASSES of them), so a
//     DSv4 row (192 q chunks + 64 kv chunks) is exactly two 16-byte loads per
//     thread, coalesced, from strided split views as well as contiguous rows;
//   * the thread's gamma chunks are loaded once, as fp32, and the next row's
//     chunks are loaded while the current row is reduced and stored;
//   * the two sums of squares are reduced with warp shuffles and one
//     cross-warp step through shared memory (double-buffered by row parity,
//     so one barrier per row suffices);
//   * Kq is a multiple of 128, so in every pass each aligned half-warp holds
//     exactly one 128-column q group (or kv, or nothing): the group amax is a
//     4-step 16-lane shuffle, and lane 0 of the half-warp stores the scale;
//   * elementwise fp32 work uses the packed f32x2 instructions of sm_100+;
//   * codes are packed 8 per thread and stored as one 8-byte word, kv as one
//     16-byte word.
// Each input byte is read once and each output byte written once.

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "debug_check.cuh"
#include "dsnq_internal.h"
#include "group_quant.cuh"

namespace dsnq {

constexpr int kThreads = 128;       // one warp-group per row
constexpr int kChunk = 8;           // bf16 per 16-byte chunk
// CTAs per SM the register budget of the warp-group-per-row kernel is sized
// for (64 registers per thread up to two chunks per thread, 128 beyond).
__host__ __device__ constexpr int min_blocks_per_sm(int passes) { return passes <= 2 ? 8 : 4; }

enum Mode : int {
    kFused = 0,      // q -> fp8 codes + scales, kv -> bf16
    kNormOnly = 1,   // q -> bf16, kv -> bf16 (baseline step 1)
    kQuantOnly = 2,  // x (passed as q) -> fp8 codes + scales, no norm (baseline step 2)
};

struct RowArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kv;
    const __nv_bfloat16* gamma_q;
    const __nv_bfloat16* gamma_kv;
    int64_t ldq, ldkv;
    int64_t M;
    int cq, ckv;           // chunk counts Kq/8, Kkv/8
    float kq_f, kkv_f;     // Kq and Kkv as floats (divisors of the mean)
    float eps;
    uint8_t* q_fp8;        // kFused / kQuantOnly
    __nv_bfloat16* q_bf16; // kNormOnly
    int64_t ldq_out;
    float* scale;
    int64_t scale_row_stride, scale_group_stride;  // (m, g) at m*rs + g*gs
    __nv_bfloat16* kv_out;
    int64_t ldkv_out;
    uint32_t inject;       // test hooks (dsnq_debug_set)
};

__device__ __forceinline__ uint4 pack8_bf16(const float2 (&f)[4]) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[i].x, f[i].y);
    return v;
}

// ---- the quantize step: code = e4m3_rn_satfinite(fp32(x / scale))
//
// The quotient is defined as the IEEE fp32 division x / scale.  Dividing
// every element is expensive, so each group first forms y = fp32(1/scale)
// (one correctly rounded reciprocal per group) and the approximation
// q = fp32(x * y), whose relative distance to fp32(x / scale) is below 2^-22.
// E4M3 rounding is monotone, so if q * (1 - 2^-20) and q * (1 + 2^-20) give
// the same code, that code is the code of fp32(x / scale) too; otherwise (the
// quotient sits within 2^-20 of an E4M3 rounding boundary, or the scale is
// too small for its reciprocal to be finite) the pair takes the IEEE division.
struct QuantScale {
    float scale;   // amax / 448, IEEE fp32
    float recip;   // fp32(1 / scale), 0 for an all-zero group
    bool exact;    // true: always use the division (reciprocal not finite)
};

__device__ __forceinline__ QuantScale make_quant_scale(float amax) {
    QuantScale qs;
    qs.scale = amax / kE4M3Max;                       // IEEE fp32 divide
    qs.exact = qs.scale > 0.f && qs.scale < 1.0e-36f;
    // The reciprocal only has to be within 2^-22 of 1/scale for the bracket
    // below (relative width 2^-20), which the fast divide (2 ulp) meets.
    qs.recip = (qs.scale > 0.f && !qs.exact) ? __fdividef(1.0f, qs.scale) : 0.f;
    return qs;
}

// Exact path of quant4 (rare): the IEEE division itself.
__device__ __noinline__ uint32_t quant4_exact(float2 v0, float2 v1, float scale) {
    if (scale > 0.f)
        return e4m3x2(make_float2(__fdiv_rn(v0.x, scale), __fdiv_rn(v0.y, scale))) |
               (e4m3x2(make_float2(__fdiv_rn(v1.x, scale), __fdiv_rn(v1.y, scale))) << 16);
    return e4m3x2(make_float2(v0.x * 0.f, v0.y * 0.f)) |           // all-zero group: signed zeros
           (e4m3x2(make_float2(v1.x * 0.f, v1.y * 0.f)) << 16);
}

// Four codes (little-endian bytes) of the values of the pairs v0, v1.
__device__ __forceinline__ uint32_t quant4(float2 v0, float2 v1, const QuantScale& qs) {
    const float2 y = make_float2(qs.recip, qs.recip);
    const float2 q0 = mul2(v0, y), q1 = mul2(v1, y);
    const float2 lo = make_float2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f);
    const float2 hi = make_float2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f);
    const uint32_t wlo = e4m3x2(mul2(q0, lo)) | (e4m3x2(mul2(q1, lo)) << 16);
    const uint32_t whi = e4m3x2(mul2(q0, hi)) | (e4m3x2(mul2(q1, hi)) << 16);
    if (wlo == whi && !qs.exact) return wlo;
    return quant4_exact(v0, v1, qs.scale);
}

// Eight E4M3FN codes of x / scale (x as four pairs), little-endian in a uint2.
__device__ __forceinline__ uint2 pack8_e4m3(const float2 (&f)[4], const QuantScale& qs) {
    return make_uint2(quant4(f[0], f[1], qs), quant4(f[2], f[3], qs));
}

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int MODE, int PASSES>
__global__ void __launch_bounds__(kThreads, min_blocks_per_sm(PASSES))
row_norm_quant_kernel(const RowArgs a) {
    grid_dependency_wait();      // inputs are read only once the previous kernel's writes are visible
    allow_dependent_launch();
    bounds_self_test(a.inject);
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;

    // Fixed role of each of this thread's chunks (same for every row).
    bool is_q[PASSES], live[PASSES];
    int col[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int c = p * kThreads + t;
        is_q[p] = c < a.cq;
        live[p] = c < a.cq + a.ckv;
        col[p] = (is_q[p] ? c : c - a.cq) * kChunk;
    }

    // Gamma, once per CTA, as fp32 pairs.
    float2 gm[PASSES][4];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        uint4 gr = make_uint4(0, 0, 0, 0);
        if (MODE != kQuantOnly && live[p])
            gr = __ldg(reinterpret_cast<const uint4*>((is_q[p] ? a.gamma_q : a.gamma_kv) + col[p]));
        unpack8(gr, gm[p]);
    }

    auto load_row = [&](int64_t m, uint4 (&raw)[PASSES]) {
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            raw[p] = make_uint4(0, 0, 0, 0);
            if (live[p] && bounds_ok(m < a.M && col[p] + kChunk <= (is_q[p] ? a.cq : a.ckv) * kChunk)) {
                const __nv_bfloat16* src = is_q[p] ? a.q + m * a.ldq + col[p] : a.kv + m * a.ldkv + col[p];
                raw[p] = __ldg(reinterpret_cast<const uint4*>(src));
            }
        }
    };

    __shared__ float red[2][2][kThreads / 32];   // [row parity][q, kv][warp]
    uint4 cur[PASSES];
    int64_t m = blockIdx.x;
    if (m < a.M) load_row(m, cur);
    int par = 0;
    for (; m < a.M; m += gridDim.x, par ^= 1) {
        // Prefetch the next row of this CTA while this one is processed.
        uint4 nxt[PASSES];
        const int64_t mn = m + gridDim.x;
        if (mn < a.M) load_row(mn, nxt);

        float2 x[PASSES][4];
#pragma unroll
        for (int p = 0; p < PASSES; ++p) unpack8(cur[p], x[p]);

        if (MODE != kQuantOnly) {
            float2 sq = make_float2(0.f, 0.f), skv = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 4; ++i) s2 = fma2(x[p][i], x[p][i], s2);
                if (is_q[p]) { sq.x += s2.x; sq.y += s2.y; }    // dead chunks hold zeros
                else { skv.x += s2.x; skv.y += s2.y; }
            }
            float ssq_q = warp_sum(sq.x + sq.y);
            float ssq_kv = warp_sum(skv.x + skv.y);
            if (lane == 0) { red[par][0][warp] = ssq_q; red[par][1][warp] = ssq_kv; }
            __syncthreads();
            ssq_q = (red[par][0][0] + red[par][0][1]) + (red[par][0][2] + red[par][0][3]);
            ssq_kv = (red[par][1][0] + red[par][1][1]) + (red[par][1][2] + red[par][1][3]);
            // Correctly rounded sqrt and divide (not the approximate rsqrt).
            const float r_q = 1.0f / sqrtf(ssq_q / a.kq_f + a.eps);
            const float r_kv = 1.0f / sqrtf(ssq_kv / a.kkv_f + a.eps);
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                const float r = is_q[p] ? r_q : r_kv;
                const float2 r2 = make_float2(r, r);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[p][i] = mul2(mul2(x[p][i], r2), gm[p][i]);
            }
        }

#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            // Debug build: a chunk whose indices fail the check stores nothing
            // (it still takes part in the warp's shuffles).
            const bool in = bounds_ok(m < a.M && (!live[p] || col[p] + kChunk <= (is_q[p] ? a.cq : a.ckv) * kChunk));
            if (MODE == kNormOnly) {
                if (!live[p] || !in) continue;
                if (is_q[p])
                    *reinterpret_cast<uint4*>(a.q_bf16 + m * a.ldq_out + col[p]) = pack8_bf16(x[p]);
                else
                    *reinterpret_cast<uint4*>(a.kv_out + m * a.ldkv_out + col[p]) = pack8_bf16(x[p]);
                continue;
            }
            // Group amax: every aligned half-warp of this pass holds one q group,
            // or kv / dead chunks whose result is discarded.  All lanes shuffle.
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(x[p][i].x), fabsf(x[p][i].y)));
            amax = half_warp_max(amax);
            if (!live[p] || !in) continue;
            if (is_q[p]) {
                const QuantScale qs = make_quant_scale(amax);
                *reinterpret_cast<uint2*>(a.q_fp8 + m * a.ldq_out + col[p]) = pack8_e4m3(x[p], qs);
                if ((lane & 15) == 0)
                    a.scale[m * a.scale_row_stride + (col[p] / 128) * a.scale_group_stride] = qs.scale;
            } else if (MODE == kFused) {
                *reinterpret_cast<uint4*>(a.kv_out + m * a.ldkv_out + col[p]) = pack8_bf16(x[p]);
            }
        }
#pragma unroll
        for (int p = 0; p < PASSES; ++p) cur[p] = nxt[p];
    }
}

// ---------------------------------------------------------------------------
// One warp per token row, for rows of at most 256 chunks (DSv4: 192 q + 64
// kv).  Lane l owns chunks l, l+32, ... (CPT of them); with Kq a multiple of
// 128, each aligned half-warp of chunk slot j holds one q group.  No block
// barrier per row: the row's sums of squares are warp shuffles.  Gamma lives
// in shared memory as fp32, loaded once per CTA.
// ---------------------------------------------------------------------------
constexpr int kRowWarps = 4;        // rows in flight per CTA
constexpr int kRowCtasPerSM = 4;    // register budget: up to 128 per thread

template <int MODE, int CPT>
__global__ void __launch_bounds__(kRowWarps * 32, kRowCtasPerSM)
warp_row_kernel(const RowArgs a) {
    grid_dependency_wait();      // inputs are read only once the previous kernel's writes are visible
    allow_dependent_launch();
    bounds_self_test(a.inject);
    extern __shared__ float gamma_s[];          // [Kq + Kkv] fp32
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int kq = a.cq * kChunk, width = (a.cq + a.ckv) * kChunk;

    bool is_q[CPT], live[CPT];
    int col[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int c = j * 32 + lane;
        is_q[j] = c < a.cq;
        live[j] = c < a.cq + a.ckv;
        col[j] = (is_q[j] ? c : c - a.cq) * kChunk;
    }

    auto load_row = [&](int64_t m, uint4 (&raw)[CPT]) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            raw[j] = make_uint4(0, 0, 0, 0);
            if (live[j] && bounds_ok(m < a.M && col[j] + kChunk <= (is_q[j] ? a.cq : a.ckv) * kChunk)) {
                const __nv_bfloat16* src = is_q[j] ? a.q + m * a.ldq + col[j] : a.kv + m * a.ldkv + col[j];
                raw[j] = __ldg(reinterpret_cast<const uint4*>(src));
            }
        }
    };

    const int64_t stride = static_cast<int64_t>(gridDim.x) * kRowWarps;
    int64_t m = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
    uint4 cur[CPT];
    if (m < a.M) load_row(m, cur);               // in flight while gamma is staged

    if (MODE != kQuantOnly) {
        for (int i = threadIdx.x * kChunk; i < width; i += kRowWarps * 32 * kChunk) {
            const __nv_bfloat16* gsrc = i < kq ? a.gamma_q + i : a.gamma_kv + (i - kq);
            float2 g[4];
            unpack8(__ldg(reinterpret_cast<const uint4*>(gsrc)), g);
#pragma unroll
            for (int k = 0; k < 4; ++k) reinterpret_cast<float2*>(gamma_s + i)[k] = g[k];
        }
        __syncthreads();
    }

    for (; m < a.M; m += stride) {
        uint4 nxt[CPT];
        const int64_t mn = m + stride;
        if (mn < a.M) load_row(mn, nxt);         // prefetch this warp's next row

        // The row stays packed (bf16) in registers; it is unpacked once for
        // the sums of squares and once more, chunk by chunk, for the outputs.
        float r_q = 1.f, r_kv = 1.f;
        if (MODE != kQuantOnly) {
            float2 sq = make_float2(0.f, 0.f), skv = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                float2 x[4];
                unpack8(cur[j], x);
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 4; ++i) s2 = fma2(x[i], x[i], s2);
                if (is_q[j]) { sq.x += s2.x; sq.y += s2.y; }    // dead chunks hold zeros
                else { skv.x += s2.x; skv.y += s2.y; }
            }
            const float ssq_q = warp_sum(sq.x + sq.y);
            const float ssq_kv = warp_sum(skv.x + skv.y);
            // Correctly rounded sqrt and divide (not the approximate rsqrt).
            r_q = 1.0f / sqrtf(ssq_q / a.kq_f + a.eps);
            r_kv = 1.0f / sqrtf(ssq_kv / a.kkv_f + a.eps);
        }

#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            // Debug build: a chunk whose indices fail the check stores nothing
            // (it still takes part in the warp's votes and shuffles).
            const bool in = bounds_ok(m < a.M && (!live[j] || col[j] + kChunk <= (is_q[j] ? a.cq : a.ckv) * kChunk));
            float2 x[4];
            unpack8(cur[j], x);
            if (MODE != kQuantOnly) {
                const float r = is_q[j] ? r_q : r_kv;
                const float2 r2 = make_float2(r, r);
                const float4* gp = reinterpret_cast<const float4*>(gamma_s + (is_q[j] ? 0 : kq) + col[j]);
                float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
                if (live[j]) { g0 = gp[0]; g1 = gp[1]; }
                x[0] = mul2(mul2(x[0], r2), make_float2(g0.x, g0.y));
                x[1] = mul2(mul2(x[1], r2), make_float2(g0.z, g0.w));
                x[2] = mul2(mul2(x[2], r2), make_float2(g1.x, g1.y));
                x[3] = mul2(mul2(x[3], r2), make_float2(g1.z, g1.w));
            }
            if (MODE == kNormOnly) {
                if (!live[j] || !in) continue;
                if (is_q[j])
                    *reinterpret_cast<uint4*>(a.q_bf16 + m * a.ldq_out + col[j]) = pack8_bf16(x);
                else
                    *reinterpret_cast<uint4*>(a.kv_out + m * a.ldkv_out + col[j]) = pack8_bf16(x);
                continue;
            }
            // Slots whose chunks are kv (or past the row) for the whole warp skip the group work.
            if (__any_sync(0xffffffffu, is_q[j])) {
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(x[i].x), fabsf(x[i].y)));
                amax = half_warp_max(amax);
                if (is_q[j]) {
                    if (!in) continue;
                    const QuantScale qs = make_quant_scale(amax);
                    *reinterpret_cast<uint2*>(a.q_fp8 + m * a.ldq_out + col[j]) = pack8_e4m3(x, qs);
                    if ((lane & 15) == 0)
                        a.scale[m * a.scale_row_stride + (col[j] / 128) * a.scale_group_stride] = qs.scale;
                    continue;
                }
            }
            if (MODE == kFused && live[j] && in)
                *reinterpret_cast<uint4*>(a.kv_out + m * a.ldkv_out + col[j]) = pack8_bf16(x);
        }
#pragma unroll
        for (int j = 0; j < CPT; ++j) cur[j] = nxt[j];
    }
}

// ---------------------------------------------------------------------------
// Fused warp-per-row kernel for the DSv4 row: Kq = 1536 (6 slots of 256
// columns, one 128-column group per half-warp and slot) and Kkv = 512 (2
// slots).  Lane l holds chunks l, l+32, ... of the row (16 bytes each).
//   * each slot's role is known at compile time (no per-chunk predicates);
//   * rows reach the warp through a ring of kRingRows row buffers in shared
//     memory that its lanes fill with cp.async: the warp's first kRingRows
//     rows are requested at once, and each row read out of the ring is
//     replaced by the request for the row kRingRows further on, so the loads
//     run ahead of the arithmetic by that many rows without holding
//     registers.  Each lane copies and later reads only its own chunks, so
//     its own cp.async.wait_group orders the two.  Measured on GB300 against
//     the next row held in registers (four-warp CTAs, four per SM): M=2048
//     6.65 -> 6.02 us, M=8192 14.7-15.0 -> 14.5 us, M=32768 40.2 -> 39.2 us
//     per call in a graph; three rows in flight, 16-warp CTAs, or three
//     CTAs per SM (80 registers, spills) measured slower;
//   * the work that is the same for a whole warp is done once, by the lanes
//     it concerns, and handed to the others by shuffles:
//       - the two sums of squares are reduced by a reduce-scatter (lanes
//         0-15 end with the q sum, 16-31 with the kv sum), each half takes
//         its 1/sqrt(mean + eps) in one IEEE chain, two shuffles broadcast;
//       - the twelve group maxima are reduced by a reduce-scatter over the
//         six q slots (lanes with lane bit 3 clear keep slots 0-2, set 3-5),
//         so that lane 16h + 8b + i (i < 3) holds group 2(3b + i) + h: that
//         lane alone forms the group's scale and reciprocal, stores the
//         scale, and the other lanes fetch both by shuffle;
//   * the quantize step uses bracket reciprocals scaled once per group and
//     takes the exactness decision for three slots with one warp vote.
// ---------------------------------------------------------------------------
constexpr int kFusedWarps = 8;      // warps (rows in work) per CTA
constexpr int kFusedCtasPerSM = 2;  // register budget: 128 per thread
constexpr int kRingRows = 2;        // rows in flight per warp
constexpr int kDsv4RowBytes = (6 + 2) * 256 * 2;   // one q + kv row in bf16 (4 KB)

__host__ __device__ constexpr size_t fused_smem_bytes() {
    return static_cast<size_t>(8 * 256) * sizeof(float) +
           static_cast<size_t>(kFusedWarps) * kRingRows * kDsv4RowBytes;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int QS, int KS>
__global__ void __launch_bounds__(kFusedWarps * 32, kFusedCtasPerSM)
warp_row_fused_kernel(const RowArgs a) {
    // KS = 0: the single-latent call (the q latent alone; no kv chunk is touched).
    static_assert(QS == 6 && (KS == 2 || KS == 0), "the lane roles below are laid out for the DSv4 row");
    grid_dependency_wait();      // inputs are read only once the previous kernel's writes are visible
    allow_dependent_launch();
    bounds_self_test(a.inject);
    constexpr int CPT = QS + KS;
    constexpr unsigned kAll = 0xffffffffu;
    extern __shared__ __align__(16) float gamma_s[];   // [(QS + KS) * 256] fp32: gamma_q then gamma_kv; then the rings
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    constexpr int kq = QS * 256, width = CPT * 256;
    static_assert(CPT * 256 * 2 <= kDsv4RowBytes, "ring slots hold one row");
    const bool q_half = lane < 16;              // reduce-scatter roles
    const bool hi8 = (lane & 8) != 0;
    const int gi = lane & 7;                    // group slot this lane forms (when < 3)
    const int h = lane >> 4;                    // half-warp: group 2j + h in slot j
    // This lane's 16-byte chunk of slot j of ring row r: byte r * row + j * 512 + lane * 16.
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(gamma_s + width)) +
                          static_cast<uint32_t>(warp * kRingRows * kDsv4RowBytes + lane * 16);

    // Requests row mm into ring row r (nothing past the last row); always one
    // commit group, so that the group count stays one per ring step.
    auto request_row = [&](int64_t mm, int r) {
        const bool in = bounds_ok(a.cq == QS * 32 && a.ckv == KS * 32 && r < kRingRows);
        if (mm < a.M && in) {
            const __nv_bfloat16* qrow = a.q + mm * a.ldq + lane * kChunk;
            const __nv_bfloat16* kvrow = a.kv + mm * a.ldkv + lane * kChunk;
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                cp_async16(ring + r * kDsv4RowBytes + j * 512, j < QS ? qrow + j * 256 : kvrow + (j - QS) * 256);
        }
        cp_async_commit();
    };

    const int64_t stride = static_cast<int64_t>(gridDim.x) * kFusedWarps;
    int64_t m = static_cast<int64_t>(blockIdx.x) * kFusedWarps + warp;
#pragma unroll
    for (int r = 0; r < kRingRows; ++r) request_row(m + r * stride, r);   // in flight while gamma is staged

    for (int i = threadIdx.x * kChunk; i < width; i += kFusedWarps * 32 * kChunk) {
        const __nv_bfloat16* gsrc = i < kq ? a.gamma_q + i : a.gamma_kv + (i - kq);
        float2 g[4];
        unpack8(__ldg(reinterpret_cast<const uint4*>(gsrc)), g);
#pragma unroll
        for (int k = 0; k < 4; ++k) reinterpret_cast<float2*>(gamma_s + i)[k] = g[k];
    }
    __syncthreads();

    const float kdiv = q_half ? a.kq_f : a.kkv_f;
    int r = 0;
    for (; m < a.M; m += stride) {
        cp_async_wait<kRingRows - 1>();          // this lane's chunks of row m have landed
        float2 x[CPT][4];
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(ring + r * kDsv4RowBytes + j * 512)
                         : "memory");
            unpack8(v, x[j]);
        }
        // The chunks are in registers, so the ring row can take the row
        // kRingRows steps ahead (the warp barrier orders the reads above
        // before the copies that overwrite them).
        __syncwarp();
        request_row(m + kRingRows * stride, r);
        r = r + 1 == kRingRows ? 0 : r + 1;

        // Sums of squares, then the reduce-scatter: lanes 0-15 finish the q
        // sum, lanes 16-31 the kv sum, each over the 32 lanes' partials.
        float2 sq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float2 skv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (j < QS) sq[i & 1] = fma2(x[j][i], x[j][i], sq[i & 1]);
                else skv[i & 1] = fma2(x[j][i], x[j][i], skv[i & 1]);
            }
        }
        const float pq = (sq[0].x + sq[1].x) + (sq[0].y + sq[1].y);
        const float pkv = (skv[0].x + skv[1].x) + (skv[0].y + skv[1].y);
        float ssq = (q_half ? pq : pkv) + __shfl_xor_sync(kAll, q_half ? pkv : pq, 16);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ssq += __shfl_xor_sync(kAll, ssq, o);
        // Correctly rounded division and sqrt (not the approximate rsqrt).
        const float rr = 1.0f / sqrtf(ssq / kdiv + a.eps);
        const float rq = __shfl_sync(kAll, rr, 0), rkv = __shfl_sync(kAll, rr, 16);

        // Normalize; kv goes straight out.
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int col = (j < QS ? j : j - QS) * 256 + lane * kChunk;
            const float r = j < QS ? rq : rkv;
            const float2 r2 = make_float2(r, r);
            const float4* gp = reinterpret_cast<const float4*>(gamma_s + (j < QS ? 0 : kq) + col);
            const float4 g0 = gp[0], g1 = gp[1];
            x[j][0] = mul2(mul2(x[j][0], r2), make_float2(g0.x, g0.y));
            x[j][1] = mul2(mul2(x[j][1], r2), make_float2(g0.z, g0.w));
            x[j][2] = mul2(mul2(x[j][2], r2), make_float2(g1.x, g1.y));
            x[j][3] = mul2(mul2(x[j][3], r2), make_float2(g1.z, g1.w));
            if (j >= QS && bounds_ok(m < a.M && col + kChunk <= a.ckv * kChunk))
                *reinterpret_cast<uint4*>(a.kv_out + m * a.ldkv_out + col) = pack8_bf16(x[j]);
        }

        // Group maxima: this lane's eight values per q slot, then the
        // reduce-scatter across the half-warp (slots 0-2 stay with lanes whose
        // bit 3 is clear, 3-5 with the others), then a butterfly on three.
        float am[QS];
#pragma unroll
        for (int j = 0; j < QS; ++j)
            am[j] = fmaxf(fmaxf(fmaxf(fabsf(x[j][0].x), fabsf(x[j][0].y)), fmaxf(fabsf(x[j][1].x), fabsf(x[j][1].y))),
                          fmaxf(fmaxf(fabsf(x[j][2].x), fabsf(x[j][2].y)), fmaxf(fabsf(x[j][3].x), fabsf(x[j][3].y))));
        float kmax[3];
#pragma unroll
        for (int i = 0; i < 3; ++i)
            kmax[i] = fmaxf(hi8 ? am[3 + i] : am[i], __shfl_xor_sync(kAll, hi8 ? am[i] : am[3 + i], 8));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
#pragma unroll
            for (int i = 0; i < 3; ++i) kmax[i] = fmaxf(kmax[i], __shfl_xor_sync(kAll, kmax[i], o));
        }
        // Lane 16h + 8b + i (i < 3) forms group 2(3b + i) + h; the other lanes
        // compute a copy they discard.
        const float own_scale = group_scale(gi == 0 ? kmax[0] : gi == 1 ? kmax[1] : kmax[2]);
        const float own_y = group_recip(own_scale);
        if (gi < 3) {
            const int g = 2 * (3 * (hi8 ? 1 : 0) + gi) + h;
            if (bounds_ok(g < a.cq / 16 && m < a.M))
                a.scale[m * a.scale_row_stride + g * a.scale_group_stride] = own_scale;
        }

        // Codes, three q slots at a time (fewer live registers).
        constexpr int kGrp = 3;
        static_assert(QS % kGrp == 0, "q slots in groups of three");
#pragma unroll
        for (int j0 = 0; j0 < QS; j0 += kGrp) {
            GroupQuant gq[kGrp];
            uint2 codes[kGrp];
            bool ok_all = true;
#pragma unroll
            for (int u = 0; u < kGrp; ++u) {
                const int j = j0 + u;                       // slot j: group 2j + h, formed by lane 16h + 8(j/3) + j%3
                const int src = (lane & 16) | ((j / 3) << 3) | (j % 3);
                gq[u] = group_quant_from(__shfl_sync(kAll, own_scale, src), __shfl_sync(kAll, own_y, src));
                bool ok;
                codes[u] = quant8_bracket(x[j], gq[u], ok);
                ok_all = ok_all && ok;
            }
            if (!__all_sync(kAll, ok_all)) {
#pragma unroll
                for (int u = 0; u < kGrp; ++u) {
                    bool ok;
                    quant8_bracket(x[j0 + u], gq[u], ok);
                    if (ok) continue;
                    codes[u] = quant8_divide(x[j0 + u], gq[u].scale);
                }
            }
            uint8_t* crow = a.q_fp8 + m * a.ldq_out + lane * kChunk;
#pragma unroll
            for (int u = 0; u < kGrp; ++u)
                if (bounds_ok(m < a.M && (j0 + u) * 256 + lane * kChunk + kChunk <= a.cq * kChunk))
                    *reinterpret_cast<uint2*>(crow + (j0 + u) * 256) = codes[u];
        }
    }
    cp_async_wait<0>();          // no copy outstanding when the CTA exits (rows past the end request none)
}

// The staged kernel's shared memory is above the default 48 KB limit; the
// attribute is set once per device.
template <int KS>
static bool fused_smem_ready() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(warp_row_fused_kernel<6, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(fused_smem_bytes())) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

template <int MODE>
static dsnq_status launch_rows(RowArgs a, int64_t M, cudaStream_t s) {
    a.inject = debug_inject_flags();
    const int chunks = a.cq + a.ckv;
    const int passes = (chunks + kThreads - 1) / kThreads;
    a.M = M;
    const int sms = device_sm_count();
    // Many rows: one warp per row (no block barrier per row).  Few rows: a
    // warp-group per row, which shortens each thread's dependency chain.
    const int64_t warp_row_min = sms > 0 ? static_cast<int64_t>(sms) * 8 : 2048;
    if (MODE == kFused && a.cq == 6 * 32 && (a.ckv == 2 * 32 || a.ckv == 0) && M >= warp_row_min) {
        // DSv4 rows (Kq = 1536, Kkv = 512, or the q latent alone): the
        // specialized warp-per-row kernel.
        const bool with_kv = a.ckv != 0;
        if (!(with_kv ? fused_smem_ready<2>() : fused_smem_ready<0>())) return DSNQ_ERR_CUDA;
        const int64_t rows_cap = sms > 0 ? static_cast<int64_t>(sms) * kFusedCtasPerSM : (M + kFusedWarps - 1) / kFusedWarps;
        const int64_t need = (M + kFusedWarps - 1) / kFusedWarps;
        dim3 grid(static_cast<unsigned>(need < rows_cap ? need : rows_cap)), block(kFusedWarps * 32);
        return launch_result(with_kv ? launch_kernel(warp_row_fused_kernel<6, 2>, grid, block, fused_smem_bytes(), s, a)
                                     : launch_kernel(warp_row_fused_kernel<6, 0>, grid, block, fused_smem_bytes(), s, a));
    }
    if (chunks <= 8 * 32 && M >= warp_row_min) {
        // Warp per row.  Enough CTAs to fill every SM at the register-limited occupancy.
        const int cpt = (chunks + 31) / 32;
        const int64_t rows_cap = sms > 0 ? static_cast<int64_t>(sms) * kRowCtasPerSM : (M + kRowWarps - 1) / kRowWarps;
        const int64_t need = (M + kRowWarps - 1) / kRowWarps;
        dim3 grid(static_cast<unsigned>(need < rows_cap ? need : rows_cap)), block(kRowWarps * 32);
        const size_t smem = MODE == kQuantOnly ? 0 : static_cast<size_t>(chunks) * kChunk * sizeof(float);
        cudaError_t e;
        switch (cpt) {
            case 1: e = launch_kernel(warp_row_kernel<MODE, 1>, grid, block, smem, s, a); break;
            case 2: e = launch_kernel(warp_row_kernel<MODE, 2>, grid, block, smem, s, a); break;
            case 3: e = launch_kernel(warp_row_kernel<MODE, 3>, grid, block, smem, s, a); break;
            case 4: e = launch_kernel(warp_row_kernel<MODE, 4>, grid, block, smem, s, a); break;
            case 5: e = launch_kernel(warp_row_kernel<MODE, 5>, grid, block, smem, s, a); break;
            case 6: e = launch_kernel(warp_row_kernel<MODE, 6>, grid, block, smem, s, a); break;
            case 7: e = launch_kernel(warp_row_kernel<MODE, 7>, grid, block, smem, s, a); break;
            default: e = launch_kernel(warp_row_kernel<MODE, 8>, grid, block, smem, s, a); break;
        }
        return launch_result(e);
    }
    // Wider rows: one warp-group per row.  Enough CTAs to fill every SM at the
    // register-limited occupancy; each walks its rows with a grid stride.
    const int64_t cap = sms > 0 ? static_cast<int64_t>(sms) * min_blocks_per_sm(passes) : M;
    dim3 grid(static_cast<unsigned>(M < cap ? M : cap)), block(kThreads);
    cudaError_t e;
    switch (passes) {
        case 1: e = launch_kernel(row_norm_quant_kernel<MODE, 1>, grid, block, 0, s, a); break;
        case 2: e = launch_kernel(row_norm_quant_kernel<MODE, 2>, grid, block, 0, s, a); break;
        case 3: e = launch_kernel(row_norm_quant_kernel<MODE, 3>, grid, block, 0, s, a); break;
        case 4: e = launch_kernel(row_norm_quant_kernel<MODE, 4>, grid, block, 0, s, a); break;
        default: return DSNQ_ERR_UNSUPPORTED;
    }
    return launch_result(e);
}

// ---------------------------------------------------------------------------
// 128x128 weight-block quantizer (load time).  One CTA per block, 256
// threads; thread t covers row t/2 of the block, 64 columns.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
weight_block_quant_kernel(int64_t N, int64_t K, const float* __restrict__ w, int64_t ldw,
                          uint8_t* __restrict__ out, int64_t ldo,
                          float* __restrict__ sw, int64_t ldsw, uint32_t debug_inject) {
    grid_dependency_wait();      // inputs are read only once the previous kernel's writes are visible
    allow_dependent_launch();
    bounds_self_test(debug_inject);
    const int64_t nb = blockIdx.y, kb = blockIdx.x;
    const int t = threadIdx.x;
    const int64_t row = nb * 128 + t / 2;
    const int64_t c0 = kb * 128 + (t & 1) * 64;
    const bool live = row < N && bounds_ok(c0 + 64 <= K);
    float v[64];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float4 f = live ? __ldg(reinterpret_cast<const float4*>(w + row * ldw + c0) + i)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float red[8];
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const QuantScale qs = make_quant_scale(amax);
    if (t == 0 && bounds_ok(nb * 128 < N && (kb + 1) * 128 <= K)) sw[nb * ldsw + kb] = qs.scale;
    if (!live) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // 16 codes per 16-byte store
        float2 f0[4], f1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f0[i] = make_float2(v[16 * j + 2 * i], v[16 * j + 2 * i + 1]);
            f1[i] = make_float2(v[16 * j + 8 + 2 * i], v[16 * j + 8 + 2 * i + 1]);
        }
        uint2 lo = pack8_e4m3(f0, qs), hi = pack8_e4m3(f1, qs);
        *reinterpret_cast<uint4*>(out + row * ldo + c0 + 16 * j) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
}

bool take_norm_quant_debug_word(cudaStream_t s, unsigned int* v) { return take_debug_word(s, v); }

}  // namespace dsnq

using namespace dsnq;

// Shape checks come first and M == 0 is accepted before any pointer check, so
// empty tensors (whose data pointer may be NULL) are a valid no-op.
static dsnq_status check_norm_shape(int64_t M, int64_t Kq, int64_t Kkv, float eps) {
    if (M < 0 || Kq <= 0 || Kkv <= 0) return DSNQ_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps > 3.0e38f) return DSNQ_ERR_INVALID_ARG;   // also rejects NaN
    if (Kq % 128 != 0 || Kkv % 8 != 0) return DSNQ_ERR_UNSUPPORTED;
    if ((Kq / 8 + Kkv / 8) > 4 * kThreads) return DSNQ_ERR_UNSUPPORTED;
    if (M > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    return DSNQ_OK;
}

static dsnq_status check_norm_inputs(int64_t Kq, int64_t Kkv, const void* q, int64_t ldq,
                                     const void* kv, int64_t ldkv, const void* gq, const void* gkv) {
    if (!q || !kv || !gq || !gkv) return DSNQ_ERR_INVALID_ARG;
    if (ldq < Kq || ldkv < Kkv) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(gq, 16) || !aligned(gkv, 16))
        return DSNQ_ERR_MISALIGNED;
    if (ldq % 8 || ldkv % 8) return DSNQ_ERR_MISALIGNED;
    return DSNQ_OK;
}

static void set_scale_strides(RowArgs& a, dsnq_scale_layout layout, int64_t ld) {
    if (layout == DSNQ_SCALE_ROW_MAJOR) { a.scale_row_stride = ld; a.scale_group_stride = 1; }
    else { a.scale_row_stride = 1; a.scale_group_stride = ld; }
}

extern "C" dsnq_status dsnq_fused_dual_rmsnorm_group_quant(
    int64_t M, int64_t Kq, int64_t Kkv,
    const void* q, int64_t ldq, const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv, float eps, int32_t group,
    void* q_fp8, int64_t ldq_out, float* q_scale, dsnq_scale_layout layout, int64_t ld_scale,
    void* kv_out, int64_t ldkv_out, void* stream) {
    dsnq_status st = check_norm_shape(M, Kq, Kkv, eps);
    if (st != DSNQ_OK) return st;
    if (layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (group != 128) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    st = check_norm_inputs(Kq, Kkv, q, ldq, kv, ldkv, gamma_q, gamma_kv);
    if (st != DSNQ_OK) return st;
    if (!q_fp8 || !q_scale || !kv_out) return DSNQ_ERR_INVALID_ARG;
    if (ldq_out < Kq || ldkv_out < Kkv) return DSNQ_ERR_INVALID_ARG;
    const int64_t ld = scale_ld(layout, M, Kq / 128, ld_scale);
    if (ld < 0) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(q_fp8, 8) || ldq_out % 8 || !aligned(kv_out, 16) || ldkv_out % 8 || !aligned(q_scale, 4))
        return DSNQ_ERR_MISALIGNED;
    RowArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const __nv_bfloat16*>(kv);
    a.gamma_q = static_cast<const __nv_bfloat16*>(gamma_q);
    a.gamma_kv = static_cast<const __nv_bfloat16*>(gamma_kv);
    a.ldq = ldq; a.ldkv = ldkv;
    a.cq = static_cast<int>(Kq / 8); a.ckv = static_cast<int>(Kkv / 8);
    a.kq_f = static_cast<float>(Kq); a.kkv_f = static_cast<float>(Kkv);
    a.eps = eps;
    a.q_fp8 = static_cast<uint8_t*>(q_fp8);
    a.ldq_out = ldq_out;
    a.scale = q_scale;
    set_scale_strides(a, layout, ld);
    a.kv_out = static_cast<__nv_bfloat16*>(kv_out);
    a.ldkv_out = ldkv_out;
    return launch_rows<kFused>(a, M, static_cast<cudaStream_t>(stream));
}

extern "C" dsnq_status dsnq_rmsnorm_group_quant(
    int64_t M, int64_t K, const void* x, int64_t ldx, const void* gamma, float eps, int32_t group,
    void* x_fp8, int64_t ldx_out, float* x_scale, dsnq_scale_layout layout, int64_t ld_scale, void* stream) {
    if (M < 0 || K <= 0) return DSNQ_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps > 3.0e38f) return DSNQ_ERR_INVALID_ARG;   // also rejects NaN
    if (layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (group != 128 || K % 128 != 0 || K / 8 > 4 * kThreads || M > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    if (!x || !gamma || !x_fp8 || !x_scale) return DSNQ_ERR_INVALID_ARG;
    if (ldx < K || ldx_out < K) return DSNQ_ERR_INVALID_ARG;
    const int64_t ld = scale_ld(layout, M, K / 128, ld_scale);
    if (ld < 0) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(gamma, 16) || ldx % 8 || !aligned(x_fp8, 8) || ldx_out % 8 ||
        !aligned(x_scale, 4))
        return DSNQ_ERR_MISALIGNED;
    // The fused kernels with an empty kv part (no kv chunk is ever touched).
    RowArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(x);
    a.kv = a.q;
    a.gamma_q = static_cast<const __nv_bfloat16*>(gamma);
    a.gamma_kv = a.gamma_q;
    a.ldq = ldx; a.ldkv = ldx;
    a.cq = static_cast<int>(K / 8); a.ckv = 0;
    a.kq_f = static_cast<float>(K); a.kkv_f = 1.0f;
    a.eps = eps;
    a.q_fp8 = static_cast<uint8_t*>(x_fp8);
    a.ldq_out = ldx_out;
    a.scale = x_scale;
    set_scale_strides(a, layout, ld);
    a.kv_out = nullptr;
    a.ldkv_out = 0;
    return launch_rows<kFused>(a, M, static_cast<cudaStream_t>(stream));
}

extern "C" dsnq_status dsnq_dual_rmsnorm_bf16(
    int64_t M, int64_t Kq, int64_t Kkv,
    const void* q, int64_t ldq, const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv, float eps,
    void* q_out, int64_t ldq_out, void* kv_out, int64_t ldkv_out, void* stream) {
    dsnq_status st = check_norm_shape(M, Kq, Kkv, eps);
    if (st != DSNQ_OK) return st;
    if (M == 0) return DSNQ_OK;
    st = check_norm_inputs(Kq, Kkv, q, ldq, kv, ldkv, gamma_q, gamma_kv);
    if (st != DSNQ_OK) return st;
    if (!q_out || !kv_out) return DSNQ_ERR_INVALID_ARG;
    if (ldq_out < Kq || ldkv_out < Kkv) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(q_out, 16) || ldq_out % 8 || !aligned(kv_out, 16) || ldkv_out % 8)
        return DSNQ_ERR_MISALIGNED;
    RowArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const __nv_bfloat16*>(kv);
    a.gamma_q = static_cast<const __nv_bfloat16*>(gamma_q);
    a.gamma_kv = static_cast<const __nv_bfloat16*>(gamma_kv);
    a.ldq = ldq; a.ldkv = ldkv;
    a.cq = static_cast<int>(Kq / 8); a.ckv = static_cast<int>(Kkv / 8);
    a.kq_f = static_cast<float>(Kq); a.kkv_f = static_cast<float>(Kkv);
    a.eps = eps;
    a.q_bf16 = static_cast<__nv_bfloat16*>(q_out);
    a.ldq_out = ldq_out;
    a.kv_out = static_cast<__nv_bfloat16*>(kv_out);
    a.ldkv_out = ldkv_out;
    return launch_rows<kNormOnly>(a, M, static_cast<cudaStream_t>(stream));
}

extern "C" dsnq_status dsnq_group_quant_bf16(
    int64_t M, int64_t K, const void* x, int64_t ldx, int32_t group,
    void* x_fp8, int64_t ldx_out, float* x_scale, dsnq_scale_layout layout, int64_t ld_scale,
    void* stream) {
    if (M < 0 || K <= 0) return DSNQ_ERR_INVALID_ARG;
    if (layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (group != 128 || K % 128 != 0 || K / 8 > 4 * kThreads) return DSNQ_ERR_UNSUPPORTED;
    if (M > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    if (!x || !x_fp8 || !x_scale) return DSNQ_ERR_INVALID_ARG;
    if (ldx < K || ldx_out < K) return DSNQ_ERR_INVALID_ARG;
    const int64_t ld = scale_ld(layout, M, K / 128, ld_scale);
    if (ld < 0) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || ldx % 8 || !aligned(x_fp8, 8) || ldx_out % 8 || !aligned(x_scale, 4))
        return DSNQ_ERR_MISALIGNED;
    RowArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(x);
    a.ldq = ldx;
    a.cq = static_cast<int>(K / 8); a.ckv = 0;
    a.q_fp8 = static_cast<uint8_t*>(x_fp8);
    a.ldq_out = ldx_out;
    a.scale = x_scale;
    set_scale_strides(a, layout, ld);
    return launch_rows<kQuantOnly>(a, M, static_cast<cudaStream_t>(stream));
}

extern "C" dsnq_status dsnq_quantize_weight_block128(
    int64_t N, int64_t K, const float* w, int64_t ldw, void* w_fp8, int64_t ldw_out,
    float* w_scale, int64_t ld_wscale, void* stream) {
    if (N < 0 || K <= 0) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0) return DSNQ_ERR_UNSUPPORTED;
    if (N == 0) return DSNQ_OK;
    if (!w || !w_fp8 || !w_scale) return DSNQ_ERR_INVALID_ARG;
    if (ldw < K || ldw_out < K || ld_wscale < K / 128) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(w, 16) || ldw % 4 || !aligned(w_fp8, 16) || ldw_out % 16 || !aligned(w_scale, 4))
        return DSNQ_ERR_MISALIGNED;
    const int64_t nb = (N + 127) / 128;
    if (nb > 65535) return DSNQ_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(nb));
    return launch_result(launch_kernel(weight_block_quant_kernel, grid, dim3(256), 0,
                                       static_cast<cudaStream_t>(stream), N, K, w, ldw,
                                       static_cast<uint8_t*>(w_fp8), ldw_out, w_scale, ld_wscale,
                                       debug_inject_flags()));
}
