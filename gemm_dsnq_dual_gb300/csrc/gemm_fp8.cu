// W8A8 block-scaled FP8 GEMM on pre-quantized activations, tcgen05 + TMA +
// TMEM, for one or two consumers of the same activation.
//
//   out[m, n] = bf16( sum_kb sa(m, kb) * sw[n/128, kb] * sum_{k in kb} a[m,k] w[n,k] )
//
// Method: vLLM PR #53540 (prhub summary, rocm.py snippet
// apply_pre_quantized_block_scaled_mm: the fused quant's (fp8, per-1x128
// scale) pair drives the block-scaled GEMM directly, A=x_fp8, As=x_scale,
// B=weight, Bs=weight_scale) and sglang PR #27289 (aiter_w8a8_block_fp8_linear,
// block_size [128, 128], the input_scale branch, bf16 output).
//
// Design (GB300, sm_103a):
//   * The contraction runs on the 5th-generation tensor cores:
//     tcgen05.mma.kind::f8f6f4 (E4M3 x E4M3 -> fp32) with both operands
//     K-major in shared memory (128-byte swizzle), fed by TMA
//     (cp.async.bulk.tensor) through a STAGES-deep mbarrier ring.
//   * One pipeline stage is one 128-wide K block, i.e. exactly one scale
//     block.  The activation scale differs per row and per K block, so it
//     cannot be folded into the MMA: each K block is accumulated from zero into
//     one of two TMEM buffers, and the promotion warps read it back
//     (tcgen05.ld), multiply by sa * sw and add it into fp32 registers while the
//     MMA of the next K block fills the other buffer.
//   * Warp roles: warp 0 issues TMA, warp 1 allocates TMEM and issues MMA
//     (one elected lane), warps 2..9 promote and store.  Warp w may only read
//     TMEM lanes 32*(w%4)..+31, so warps 2..5 and 6..9 each cover all 128 lanes
//     and split the tile's columns in two halves.
//   * Orientation.  The MMA's M side ("P", 128 rows) and N side ("Q", BN rows)
//     are either (activations, weights) for large M, or (weights, activations)
//     for decode batches (swap-AB): 128 weight rows then fill the MMA rows and
//     the few tokens become the MMA's N of 16..64, so no tensor-core row is
//     wasted on padding and the kernel streams the weights.
//   * Dual consumer: the tile index space of both problems is concatenated
//     into one launch; both read the same activation tensor map.
//   * Every wait is bounded (globaltimer); on expiry the kernel records a
//     timeout in the device status word, drains its own copies and MMAs with
//     bounded waits, frees its TMEM and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dsnq_internal.h"

namespace dsnq {
namespace gemm {

constexpr int kBK = 128;            // K bytes per stage = one scale block
constexpr int kUmmaK = 32;          // K per tcgen05.mma kind::f8f6f4
constexpr int kPRows = 128;         // MMA M
constexpr uint32_t kStatusTimeout = 1u;

__device__ unsigned int g_status;   // device status word (bit 0: a wait timed out)

struct Problem {
    int N;
    int tiles_n;
    const float* w_scale;
    int64_t ld_ws;
    __nv_bfloat16* out;
    int64_t ldo;
};

struct Params {
    int M, K, KB;
    const float* a_scale;
    int64_t as_rs, as_gs;          // sa(m, g) = a_scale[m * as_rs + g * as_gs]
    int tiles_m;                   // tiles along the activation rows
    int tiles0;                    // tiles of problem 0
    int total_tiles;               // tiles of both problems
    Problem prob[2];
    uint64_t timeout_ns;
    uint32_t inject;
};

// ----------------------------------------------------------------- PTX glue

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Gives up when another
// thread of the CTA has raised *abort, or after timeout_ns, in which case it
// raises *abort and records the timeout in the device status word.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (now_ns() - t0 > timeout_ns) {
            *abort = 1;
            atomicOr(&g_status, kStatusTimeout);
            return false;
        }
    }
}

// Drain wait: bounded by time only (used after an abort, to let this CTA's own
// copies and MMAs land before its shared and tensor memory are released).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = now_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (now_ns() - t0 > timeout_ns) return;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> fp32.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x N consecutive 32-bit TMEM columns; thread i gets lane (base+i).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr));
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart
// (stride byte offset), leading byte offset unused for this layout,
// descriptor version 1, layout code 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>(1) << 16;                 // LBO (ignored), 16 bytes
    d |= static_cast<uint64_t>((1024 >> 4) & 0x3FFF) << 32;  // SBO
    d |= static_cast<uint64_t>(1) << 46;                 // version
    d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f8f6f4: D fp32, A and B E4M3, both K-major,
// MMA shape 128 x BN.
__host__ __device__ constexpr uint32_t idesc_e4m3(int bn) {
    return (1u << 4)                                   // D format fp32
           | (0u << 7) | (0u << 10)                    // A, B = E4M3
           | (static_cast<uint32_t>(bn >> 3) << 17)    // N >> 3
           | (static_cast<uint32_t>(kPRows >> 4) << 24);  // M >> 4
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------- kernel

// Compile-time shape of one kernel variant.
//   BN        MMA N (rows of the Q operand per tile)
//   SWAP      false: P = activations, Q = weights; true: P = weights, Q = activations
//   STAGES    depth of the shared-memory ring (one 128-wide K block per stage)
//   NBUF      TMEM partial-sum buffers (the MMA may run NBUF-1 K blocks ahead)
//   EPI_WARPS promotion warps (a multiple of 4: one per TMEM lane quarter and slice)
template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS>
struct Cfg {
    static constexpr int kPBytes = kPRows * kBK;       // 16 KB
    static constexpr int kQBytes = BN * kBK;
    static constexpr int kStageBytes = kPBytes + kQBytes;
    static constexpr int kTmemNeed = NBUF * BN;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                     : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kSlices = EPI_WARPS / 4;       // column slices per lane quarter
    static constexpr int kCols = BN / kSlices;          // tile columns per promotion thread
    static constexpr int kLd = kCols >= 64 ? 32 : (kCols >= 16 ? 16 : kCols);  // columns per tcgen05.ld
    static constexpr int kThreads = (2 + EPI_WARPS) * 32;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128 is 16..256 step 16");
    static_assert(kTmemNeed <= 512, "TMEM holds 512 fp32 columns");
    static_assert(EPI_WARPS % 4 == 0 && BN % kSlices == 0, "promotion warps tile the accumulator");
    static_assert(kCols % 8 == 0 && kCols % kLd == 0, "TMEM is read 8 columns at a time at least");
    // Non-swap: a thread's columns must share one 128-feature weight-scale block.
    static_assert(SWAP || (kPRows % kCols == 0), "non-swap slices stay inside a scale block");
};

// Tile t of the concatenated tile space -> (problem, first activation row, first feature).
// Activation tiles vary fastest, so CTAs running together share weight tiles in L2.
template <int BN, bool SWAP>
__device__ __forceinline__ void tile_coords(const Params& p, int t, int& pi, int& m0, int& n0) {
    pi = t < p.tiles0 ? 0 : 1;
    if (pi) t -= p.tiles0;
    const int tm = t % p.tiles_m, tn = t / p.tiles_m;
    m0 = SWAP ? tm * BN : tm * kPRows;
    n0 = SWAP ? tn * kPRows : tn * BN;
}

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS>
__global__ void __launch_bounds__(Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS>::kThreads, 1)
block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_w0,
                         const __grid_constant__ CUtensorMap map_w1,
                         const Params p) {
    using C = Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled tiles.
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    uint64_t* full = bars;                    // [STAGES] TMA -> MMA
    uint64_t* empty = bars + STAGES;          // [STAGES] MMA -> TMA
    uint64_t* tfull = bars + 2 * STAGES;      // [NBUF]   MMA -> promotion
    uint64_t* tempty = tfull + NBUF;          // [NBUF]   promotion -> MMA
    uint64_t* drain = tempty + NBUF;          // [1]      abort drain of MMAs
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* sq = reinterpret_cast<float*>(tmem_holder + 4);  // swap: [KB][BN] combined scales

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = p.total_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), EPI_WARPS);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_w0);
        tma_prefetch_desc(&map_w1);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (one lane)
        if (lane == 0) {
            uint32_t g = 0;  // K blocks of this CTA so far, across tiles
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int pi, m0, n0;
                tile_coords<BN, SWAP>(p, t, pi, m0, n0);
                const CUtensorMap* map_w = pi ? &map_w1 : &map_w0;
                const CUtensorMap* map_p = SWAP ? map_w : &map_a;
                const CUtensorMap* map_q = SWAP ? &map_a : map_w;
                const int p_row = SWAP ? n0 : m0;
                const int q_row = SWAP ? m0 : n0;
                for (int kb = 0; kb < p.KB; ++kb, ++g) {
                    const int s = g % STAGES;
                    if (!wait_bounded(smem_u32(&empty[s]), ((g / STAGES) & 1) ^ 1, abort_flag, tmo)) {
                        ok = false;
                        break;
                    }
                    if ((p.inject & 1u) && g == 0) continue;   // test hook: never arrive on full[0]
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, C::kStageBytes);
                    uint8_t* st = tiles + s * C::kStageBytes;
                    tma_load_2d(smem_u32(st), map_p, fb, kb * kBK, p_row);
                    tma_load_2d(smem_u32(st + C::kPBytes), map_q, fb, kb * kBK, q_row);
                }
            }
            if (!ok || *abort_flag) {
                // Let the copies already issued land before the CTA exits.
                const uint32_t first = g > STAGES ? g - STAGES : 0;
                for (uint32_t j = first; j < g; ++j) {
                    if ((p.inject & 1u) && j == 0) continue;
                    wait_drain(smem_u32(&full[j % STAGES]), (j / STAGES) & 1, tmo);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one lane)
        constexpr uint32_t idesc = idesc_e4m3(BN);
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.KB; ++kb, ++g) {
                    const int s = g % STAGES;
                    const int b = g % NBUF;
                    if (!wait_bounded(smem_u32(&full[s]), (g / STAGES) & 1, abort_flag, tmo) ||
                        !wait_bounded(smem_u32(&tempty[b]), ((g / NBUF) & 1) ^ 1, abort_flag, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t pa = smem_u32(tiles + s * C::kStageBytes);
                    const uint32_t qa = pa + C::kPBytes;
                    const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        tc_mma_f8(d, smem_desc_k_sw128(pa + k * kUmmaK), smem_desc_k_sw128(qa + k * kUmmaK),
                                  idesc, k > 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty[s]));    // stage free once these MMAs have read it
                    tc_commit(smem_u32(&tfull[b]));    // partial sum ready
                    any = true;
                }
            }
            if (*abort_flag && any) {
                tc_commit(smem_u32(drain));            // completes once every MMA above has
                wait_drain(smem_u32(drain), 0, tmo);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ promotion + store
        const int ew = warp - 2;                 // 0 .. EPI_WARPS-1
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int slice = ew >> 2;               // column slice of the tile
        const int row = quarter * 32 + lane;     // P row (TMEM lane)
        const int col0 = slice * C::kCols;
        uint32_t g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            int pi, m0, n0;
            tile_coords<BN, SWAP>(p, t, pi, m0, n0);
            const Problem pr = pi ? p.prob[1] : p.prob[0];
            if (SWAP) {
                // Combined scale sa(m0+j, kb) * sw[n0/128, kb] for every token j of the tile.
                named_bar_sync(1, EPI_WARPS * 32);     // previous tile's readers are done
                const int nb = n0 / kPRows;
                for (int i = threadIdx.x - 64; i < p.KB * BN; i += EPI_WARPS * 32) {
                    const int kb = i / BN, j = i % BN;
                    const int m = m0 + j;
                    float v = 0.f;
                    if (m < p.M) v = p.a_scale[m * p.as_rs + kb * p.as_gs] * pr.w_scale[nb * pr.ld_ws + kb];
                    sq[i] = v;
                }
                named_bar_sync(1, EPI_WARPS * 32);
            }

            float acc[C::kCols];
#pragma unroll
            for (int j = 0; j < C::kCols; ++j) acc[j] = 0.f;
            const int m_row = m0 + row;                       // non-swap: token of this thread
            const int nb_ns = (n0 + col0) / kPRows;           // non-swap: scale block of the slice

            for (int kb = 0; kb < p.KB; ++kb, ++g) {
                const int b = g % NBUF;
                float srow = 0.f;
                if (!SWAP && m_row < p.M)
                    srow = p.a_scale[m_row * p.as_rs + kb * p.as_gs] * pr.w_scale[nb_ns * pr.ld_ws + kb];
                // Every lane polls (each acquires the phase); the outcome is made
                // warp-uniform before the warp-collective TMEM loads.
                const bool got = wait_bounded(smem_u32(&tfull[b]), (g / NBUF) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(b * BN + col0);
#pragma unroll
                for (int c = 0; c < C::kCols; c += C::kLd) {
                    uint32_t r[C::kLd];
                    tmem_ld<C::kLd>(taddr + c, r);
                    tmem_ld_wait();
                    if (c + C::kLd == C::kCols) {
                        // Last read of this buffer: hand it back to the MMA warp.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&tempty[b]));
                    }
#pragma unroll
                    for (int j = 0; j < C::kLd; ++j) {
                        const float sc = SWAP ? sq[kb * BN + col0 + c + j] : srow;
                        acc[c + j] = fmaf(__uint_as_float(r[j]), sc, acc[c + j]);
                    }
                }
            }
            if (!ok) break;

            if (!SWAP) {
                if (m_row < p.M) {
                    __nv_bfloat16* dst = pr.out + static_cast<int64_t>(m_row) * pr.ldo + n0 + col0;
#pragma unroll
                    for (int c = 0; c < C::kCols; c += 8) {
                        if (n0 + col0 + c < pr.N) {
                            uint4 v;
                            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                h[i] = __floats2bfloat162_rn(acc[c + 2 * i], acc[c + 2 * i + 1]);
                            *reinterpret_cast<uint4*>(dst + c) = v;
                        }
                    }
                }
            } else {
                const int n = n0 + row;
                if (n < pr.N) {
#pragma unroll
                    for (int j = 0; j < C::kCols; ++j) {
                        const int m = m0 + col0 + j;
                        if (m < p.M) pr.out[static_cast<int64_t>(m) * pr.ldo + n] = __float2bfloat16_rn(acc[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::kTmemCols)
                     : "memory");
    }
}

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS>
constexpr size_t smem_bytes(int KB) {
    using C = Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS>;
    return 1024 /* alignment slack */ + STAGES * C::kStageBytes + (2 * STAGES + 2 * NBUF + 1) * 8 + 16 +
           (SWAP ? static_cast<size_t>(KB) * BN * 4 : 0);
}

}  // namespace gemm

// --------------------------------------------------------------------- host

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map over a K-major e4m3 matrix [rows, K] with row stride ld bytes; box
// = 128 bytes of K x box_rows rows, 128-byte swizzle, zero fill past the end.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t ld, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(gemm::kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::atomic<uint32_t> g_inject{0};
std::atomic<uint64_t> g_timeout_ns{0};
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

struct Consumer {
    int64_t N;
    const void* w;
    int64_t ldw;
    const float* ws;
    int64_t ldws;
    void* out;
    int64_t ldo;
};

dsnq_status check_consumer(const Consumer& c, int64_t K) {
    if (c.N < 0) return DSNQ_ERR_INVALID_ARG;
    if (c.N == 0) return DSNQ_OK;
    if (!c.w || !c.ws || !c.out) return DSNQ_ERR_INVALID_ARG;
    if (c.ldw < K || c.ldo < c.N || c.ldws < K / 128) return DSNQ_ERR_INVALID_ARG;
    if (c.N % 16 != 0) return DSNQ_ERR_UNSUPPORTED;
    if (c.N > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    if (!aligned(c.w, 16) || c.ldw % 16 || !aligned(c.out, 16) || c.ldo % 8 || !aligned(c.ws, 4))
        return DSNQ_ERR_MISALIGNED;
    return DSNQ_OK;
}

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS>
dsnq_status launch(gemm::Params& prm, const CUtensorMap& ma, const CUtensorMap& mw0, const CUtensorMap& mw1,
                   cudaStream_t stream) {
    using C = gemm::Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS>;
    auto kern = gemm::block_scaled_gemm_kernel<BN, SWAP, STAGES, NBUF, EPI_WARPS>;
    const size_t smem = gemm::smem_bytes<BN, SWAP, STAGES, NBUF, EPI_WARPS>(prm.KB);
    if (smem > 227 * 1024) return DSNQ_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
        cudaGetLastError();
        return DSNQ_ERR_CUDA;
    }
    // Persistent: one CTA per SM (the shared-memory ring allows one), each
    // walking the tile space with a stride of the grid size.
    const int sms = device_sm_count();
    const int grid = prm.total_tiles < sms ? prm.total_tiles : (sms > 0 ? sms : prm.total_tiles);
    kern<<<grid, C::kThreads, smem, stream>>>(ma, mw0, mw1, prm);
    return launch_status();
}

dsnq_status run_gemm(int64_t M, int64_t K, const void* a, int64_t lda, const float* as,
                     dsnq_scale_layout layout, int64_t ld_as, const Consumer& c0, const Consumer& c1,
                     void* stream) {
    if (M < 0 || K <= 0 || c0.N < 0 || c1.N < 0) return DSNQ_ERR_INVALID_ARG;
    if (layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0) return DSNQ_ERR_UNSUPPORTED;
    if (M > 0x7fffffffLL || K > (1LL << 20)) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;          // empty activations may come with NULL pointers
    if (!a || !as) return DSNQ_ERR_INVALID_ARG;
    if (lda < K) return DSNQ_ERR_INVALID_ARG;
    const int64_t KB = K / 128;
    const int64_t ld = scale_ld(layout, M, KB, ld_as);
    if (ld < 0) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(a, 16) || lda % 16 || !aligned(as, 4)) return DSNQ_ERR_MISALIGNED;
    dsnq_status st = check_consumer(c0, K);
    if (st != DSNQ_OK) return st;
    st = check_consumer(c1, K);
    if (st != DSNQ_OK) return st;
    if (c0.N == 0 && c1.N == 0) return DSNQ_OK;

    // Decode batches (M <= 64): swap-AB, the tokens are the MMA's N.
    // Otherwise 128x128 tiles with four TMEM partial buffers.
    const bool swap = M <= 64;
    const int bn = swap ? (M <= 16 ? 16 : M <= 32 ? 32 : 64) : 128;
    const int a_box = swap ? bn : gemm::kPRows;
    const int w_box = swap ? gemm::kPRows : bn;

    gemm::Params prm{};
    prm.M = static_cast<int>(M);
    prm.K = static_cast<int>(K);
    prm.KB = static_cast<int>(KB);
    prm.a_scale = as;
    if (layout == DSNQ_SCALE_ROW_MAJOR) { prm.as_rs = ld; prm.as_gs = 1; }
    else { prm.as_rs = 1; prm.as_gs = ld; }
    const int64_t rows_per_a_tile = swap ? bn : gemm::kPRows;
    prm.tiles_m = static_cast<int>((M + rows_per_a_tile - 1) / rows_per_a_tile);

    CUtensorMap ma, mw[2];
    if (!make_map(&ma, a, M, K, lda, a_box)) return DSNQ_ERR_CUDA;
    const Consumer* cs[2] = {&c0, &c1};
    int64_t total = 0;
    int np = 0;
    for (int i = 0; i < 2; ++i) {
        const Consumer& c = *cs[i];
        if (c.N == 0) continue;
        gemm::Problem& pr = prm.prob[np];
        pr.N = static_cast<int>(c.N);
        const int64_t feat_per_tile = swap ? gemm::kPRows : bn;
        pr.tiles_n = static_cast<int>((c.N + feat_per_tile - 1) / feat_per_tile);
        pr.w_scale = c.ws;
        pr.ld_ws = c.ldws;
        pr.out = static_cast<__nv_bfloat16*>(c.out);
        pr.ldo = c.ldo;
        if (!make_map(&mw[np], c.w, c.N, K, c.ldw, w_box)) return DSNQ_ERR_CUDA;
        const int64_t tiles = static_cast<int64_t>(prm.tiles_m) * pr.tiles_n;
        if (np == 0) prm.tiles0 = static_cast<int>(tiles);
        total += tiles;
        ++np;
    }
    if (np == 1) mw[1] = mw[0];
    if (total > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    prm.total_tiles = static_cast<int>(total);
    const uint64_t tmo = g_timeout_ns.load();
    prm.timeout_ns = tmo ? tmo : kDefaultTimeoutNs;
    prm.inject = g_inject.load();

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (bn) {
        case 16: return launch<16, true, 8, 4, 8>(prm, ma, mw[0], mw[1], s);
        case 32: return launch<32, true, 8, 4, 8>(prm, ma, mw[0], mw[1], s);
        case 64: return launch<64, true, 8, 4, 8>(prm, ma, mw[0], mw[1], s);
        default: return launch<128, false, 6, 4, 8>(prm, ma, mw[0], mw[1], s);
    }
}

}  // namespace
}  // namespace dsnq

using namespace dsnq;

extern "C" dsnq_status dsnq_block_scaled_fp8_gemm(int64_t M, int64_t N, int64_t K, const void* a_fp8, int64_t lda,
                                                 const float* a_scale, dsnq_scale_layout a_scale_layout,
                                                 int64_t ld_ascale, const void* w_fp8, int64_t ldw,
                                                 const float* w_scale, int64_t ld_wscale, void* out_bf16,
                                                 int64_t ldo, void* stream) {
    Consumer c0{N, w_fp8, ldw, w_scale, ld_wscale, out_bf16, ldo};
    Consumer c1{0, nullptr, 0, nullptr, 0, nullptr, 0};
    return run_gemm(M, K, a_fp8, lda, a_scale, a_scale_layout, ld_ascale, c0, c1, stream);
}

extern "C" dsnq_status dsnq_block_scaled_fp8_gemm_dual(
    int64_t M, int64_t K, const void* a_fp8, int64_t lda, const float* a_scale, dsnq_scale_layout a_scale_layout,
    int64_t ld_ascale, int64_t N1, const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale,
    void* out1_bf16, int64_t ldo1, int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale,
    int64_t ld_w2scale, void* out2_bf16, int64_t ldo2, void* stream) {
    Consumer c0{N1, w1_fp8, ldw1, w1_scale, ld_w1scale, out1_bf16, ldo1};
    Consumer c1{N2, w2_fp8, ldw2, w2_scale, ld_w2scale, out2_bf16, ldo2};
    return run_gemm(M, K, a_fp8, lda, a_scale, a_scale_layout, ld_ascale, c0, c1, stream);
}

extern "C" dsnq_status dsnq_debug_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, gemm::g_status, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DSNQ_ERR_CUDA;
    }
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(gemm::g_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DSNQ_ERR_CUDA;
    }
    return (v & gemm::kStatusTimeout) ? DSNQ_ERR_TIMEOUT : DSNQ_OK;
}

extern "C" void dsnq_debug_set(uint32_t inject_flags, uint64_t wait_timeout_ns) {
    g_inject.store(inject_flags);
    g_timeout_ns.store(wait_timeout_ns);
}
