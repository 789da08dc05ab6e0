// W8A8 block-scaled FP8 GEMM on pre-quantized activations, tcgen05 + TMA +
// TMEM, for one or two consumers of the same activation; and, for a few
// decode rows, the same GEMM on bf16 activations that the kernel quantizes
// (or normalizes and quantizes) itself in its prologue.
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
//     one of NBUF TMEM buffers, and the promotion warps read it back
//     (tcgen05.ld), multiply by sa * sw and add it into fp32 registers while
//     the MMAs of the next K blocks fill the other buffers.
//   * Warp roles: warp 0 issues TMA, warp 1 allocates TMEM and issues MMA
//     (the whole warp runs the loop, one elected lane issues), warp 2 idles
//     (in the CTA-pair kernel it issues the output stores),
//     warp 3 loads the scales, warps 4.. promote and store.  The MMA warp
//     itself waits for "stage loaded" and "TMEM buffer free".  A separate gate
//     thread that waited on those and published a count of ready K blocks
//     measured slower on GB300 at every batch size: the extra hop lengthens
//     the MMA -> promotion -> MMA round trip.  Warp w may only read TMEM lanes
//     32*(w%4)..+31, so each group of four promotion warps covers all 128 lanes
//     and the groups split the tile's columns.
//   * Orientation.  The MMA's M side ("P", 128 rows) and N side ("Q", BN rows)
//     are either (activations, weights) for large M, or (weights, activations)
//     for decode batches (swap-AB): 128 weight rows then fill the MMA rows and
//     the few tokens become the MMA's N of 16..64, so no tensor-core row is
//     wasted on padding and the kernel streams the weights.
//   * Dual consumer: the tile index space of both problems is concatenated
//     into one launch; both read the same activation tensor map.
//   * bf16 activations (decode variant AQ = 1, or 2 with an RMSNorm first):
//     warps 2.. quantize the rows into a resident shared-memory operand before
//     taking up their roles, and the ring carries only the weights.
//   * Every wait is bounded (globaltimer); on expiry the kernel records a
//     timeout in the device status word, drains its own copies and MMAs with
//     bounded waits, frees its TMEM and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <tuple>
#include <vector>

#include "debug_check.cuh"
#include "dsnq_internal.h"
#include "group_quant.cuh"

namespace dsnq {
namespace gemm {

constexpr int kBK = 128;            // K bytes per stage = one scale block
constexpr int kUmmaK = 32;          // K per tcgen05.mma kind::f8f6f4
constexpr int kPRows = 128;         // MMA M
__device__ unsigned int g_status;   // device status word (kStatusTimeout: a wait timed out)

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
    int tiles_m2;                  // CTA-pair kernel: 256-row tiles along the activations
    int super0;                    // CTA-pair kernel: 256 x 256 tiles of problem 0
    int total_super;               // CTA-pair kernel: 256 x 256 tiles of both problems
    int vec_scales;                // column-major scales whose columns are 16-byte aligned
    Problem prob[2];
    uint64_t timeout_ns;
    uint32_t inject;
    const __nv_bfloat16* a_bf16;   // activations quantized in the kernel (decode, bf16 input)
    int64_t lda_bf16;
    // In-kernel RMSNorm of those activations (AQ == 2) and its side outputs,
    // written by CTA 0: kv_out, and optionally the codes and scales.
    const __nv_bfloat16* gamma_q;
    const __nv_bfloat16* kv;
    const __nv_bfloat16* gamma_kv;
    int64_t ldkv;
    int kkv;
    float kq_f, kkv_f, eps;
    __nv_bfloat16* kv_out;
    int64_t ldkv_out;
    uint8_t* q_out;                // [M, K] e4m3, row stride K (NULL: not written)
    float* qs_out;                 // [M, K/128] column-major, ld M (NULL: not written)
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

// try_wait that lets the hardware suspend the thread until the phase
// completes or `hint_ns` passes, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kSleepHintNs = 100000;   // re-check abort/timeout at least every 100 us

// Bounded wait for the phase of `parity` to complete.  Gives up when another
// thread of the CTA has raised *abort, or after timeout_ns, in which case it
// raises *abort and records the timeout in the device status word.  SPIN
// polls (lowest wake-up latency, for the waits on the MMA <-> promotion
// ring); otherwise the thread sleeps in hardware between polls.
template <bool SPIN = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    uint32_t n = 0;
    while (true) {
        if (SPIN ? mbar_try_wait(bar, parity) : mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (SPIN && (++n & 63)) continue;       // check abort and the clock every 64 polls
        
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
    while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
        if (now_ns() - t0 > timeout_ns) return;
    }
}

// Lets `ns` nanoseconds pass (abort path only): long enough for any bulk
// copy already issued to land, when there is no barrier this thread can
// watch for it.
constexpr uint64_t kAbortSettleNs = 200000;
__device__ __forceinline__ void settle_ns(uint64_t ns) {
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < ns) __nanosleep(1000);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Tiled bulk store shared -> global (rows past the tensor's extent are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Tiled bulk prefetch of a tensor tile into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// K blocks of weight tiles a decode CTA prefetches into L2 before waiting
// for the previous kernel of its stream (16 KB each).
constexpr int kPrefetchKBlocks = 24;

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA-issuing code runs converged in a whole warp (warp-uniform values,
// so they can live in uniform registers); one elected lane issues each
// tcgen05 instruction.  Issuing from a divergent single lane measured about
// 1.5x slower per K block on GB300.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> fp32 (elected lane).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x N consecutive 32-bit TMEM columns, returned as N/2 column pairs
// (64-bit registers, ready for the paired f32x2 instructions); thread i gets
// lane (base+i).  Includes the wait for the load to complete.
template <int N>
__device__ __forceinline__ void tmem_ld_pairs(uint32_t taddr, uint64_t (&r)[N / 2]);

template <>
__device__ __forceinline__ void tmem_ld_pairs<8>(uint32_t taddr, uint64_t (&r)[4]) {
    asm volatile(
        "{\n\t.reg .b32 t<8>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {t0, t1, t2, t3, t4, t5, t6, t7}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_pairs<16>(uint32_t taddr, uint64_t (&r)[8]) {
    asm volatile(
        "{\n\t.reg .b32 t<16>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7])
        : "r"(taddr)
        : "memory");
}

// Split form for software pipelining: the load is issued by one statement and
// completed by another, which takes the destination registers as operands so
// that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_pairs<32>(uint32_t taddr, uint64_t (&r)[16]) {
    asm volatile(
        "{\n\t.reg .b32 t<32>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_pairs<64>(uint32_t taddr, uint64_t (&r)[32]) {
    asm volatile(
        "{\n\t.reg .b32 t<64>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31, t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "mov.b64 %16, {t32, t33};\n\t"
        "mov.b64 %17, {t34, t35};\n\t"
        "mov.b64 %18, {t36, t37};\n\t"
        "mov.b64 %19, {t38, t39};\n\t"
        "mov.b64 %20, {t40, t41};\n\t"
        "mov.b64 %21, {t42, t43};\n\t"
        "mov.b64 %22, {t44, t45};\n\t"
        "mov.b64 %23, {t46, t47};\n\t"
        "mov.b64 %24, {t48, t49};\n\t"
        "mov.b64 %25, {t50, t51};\n\t"
        "mov.b64 %26, {t52, t53};\n\t"
        "mov.b64 %27, {t54, t55};\n\t"
        "mov.b64 %28, {t56, t57};\n\t"
        "mov.b64 %29, {t58, t59};\n\t"
        "mov.b64 %30, {t60, t61};\n\t"
        "mov.b64 %31, {t62, t63};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15]), "=l"(r[16]), "=l"(r[17]), "=l"(r[18]), "=l"(r[19]), "=l"(r[20]), "=l"(r[21]), "=l"(r[22]), "=l"(r[23]), "=l"(r[24]), "=l"(r[25]), "=l"(r[26]), "=l"(r[27]), "=l"(r[28]), "=l"(r[29]), "=l"(r[30]), "=l"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ float2 as_float2(uint64_t v) {
    float2 f;
    memcpy(&f, &v, sizeof(f));
    return f;
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

// ------------------------------------------------------------------- kernel

// Compile-time shape of one kernel variant.
//   BN        MMA N (rows of the Q operand per tile)
//   SWAP      false: P = activations, Q = weights; true: P = weights, Q = activations
//   STAGES    depth of the shared-memory ring (one 128-wide K block per stage)
//   NBUF      TMEM partial-sum buffers (the MMA may run NBUF-1 K blocks ahead)
//   EPI_WARPS promotion warps (a multiple of 4: one per TMEM lane quarter and slice)
//   AQ        (swap only) 1: the activations arrive as bf16 and are quantized
//             by the kernel into a resident shared-memory operand (the ring
//             carries only the weights); 2: the same after an RMSNorm of
//             each row, with the norm's side outputs
template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS, int AQ = 0>
struct Cfg {
    static constexpr int kPBytes = kPRows * kBK;       // 16 KB
    static constexpr int kQBytes = AQ ? 0 : BN * kBK;
    static constexpr int kStageBytes = kPBytes + kQBytes;
    // AQ: one K block of the resident operand holds kResRows rows (the few
    // live ones, then zeros).  The MMA reads BN rows from each K block's
    // base, so rows kResRows.. are the next K block's first rows (one spare
    // block after the last): garbage in token columns no call stores.
    static constexpr int kResRows = 8;
    static constexpr int kResBytes = kResRows * kBK;
    static_assert(!AQ || SWAP, "in-kernel activation quant is a decode (swap-AB) variant");
    static_assert(!AQ || (BN == 16 && kResRows * kBK == 1024), "resident K blocks on 1 KB (128-byte swizzle atoms)");
    static constexpr int kTmemNeed = NBUF * BN;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                     : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kSlices = EPI_WARPS / 4;       // column slices per lane quarter
    static constexpr int kCols = BN / kSlices;          // tile columns per promotion thread
    static constexpr int kScaleCols = SWAP ? BN : kPRows;  // activation scales per K block in a slot
    static constexpr int kScaleRegs = SWAP ? kCols / 4 : 1; // float4 of scales a thread needs per K block
    static_assert(2 * STAGES <= 32, "one producer lane per operand and stage");
    // Non-swap epilogue: each promotion warp stages its 32 x kCols bf16 block
    // (rows of kCols*2 = 64 bytes, 64-byte swizzle) for one TMA store.
    static constexpr int kStageOutBytes = SWAP ? 0 : 32 * kCols * 2;
    static_assert(SWAP || kCols == 32, "the store box is 32 rows x 64 bytes");
    static constexpr int kThreads = (4 + EPI_WARPS) * 32;  // producer, MMA, idle, scale loader, promotion
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128 is 16..256 step 16");
    static_assert(kTmemNeed <= 512, "TMEM holds 512 fp32 columns");
    static_assert(EPI_WARPS % 4 == 0 && BN % kSlices == 0, "promotion warps tile the accumulator");
    static_assert(kCols == 8 || kCols == 16 || kCols == 32 || kCols == 64, "one TMEM load per K block");
    // Non-swap: a thread's columns must share one 128-feature weight-scale block.
    static_assert(SWAP || BN == kPRows, "non-swap tiles are 128 features wide");
};

// In-kernel per-1x128 quantization of the bf16 activations (decode) into
// the resident operand: a K block's codes at a_res + kb*1024 (8 rows) in the layout
// a 128-byte-swizzled TMA copy leaves (row r's 128 codes at r*128, 16-byte
// chunk c at chunk c ^ (r & 7)); its scales to both scale slots ([kb][row],
// the second one slot_stride floats on).  Rows past M are zero (codes and
// scales, no arithmetic).  The live rows are cut into units of 256 columns
// (one row slot: a group per half-warp) spread over the nw quantizer warps,
// four units at a time per warp so that their latency chains (loads,
// shuffles, the scale division) overlap.  The arithmetic is the norm+quant
// kernels' (group_quant.cuh).
// Rows [live, 8) of the resident operand's K blocks: zero codes (whole
// 128-byte rows, so the swizzle does not matter); rows [live, BN) of the
// scales: zero.
template <int BN>
__device__ __forceinline__ void zero_rows(int KB, int live, uint8_t* a_res, float* sa_slots, int slot_stride, int qw,
                                          int nw, int lane) {
    constexpr int kRows = 8;                                // resident rows per K block
    const int zero_vec = (live < kRows ? kRows - live : 0) * (kBK / 16);   // uint4 per K block
    for (int e = qw * 32 + lane; e < KB * zero_vec; e += nw * 32) {
        const int kb = e / zero_vec, v = e % zero_vec;
        if (bounds_ok(kb < KB && live * kBK + 16 * (v + 1) <= kRows * kBK))
            reinterpret_cast<uint4*>(a_res + kb * (kRows * kBK) + live * kBK)[v] = make_uint4(0, 0, 0, 0);
    }
    for (int e = qw * 32 + lane; e < KB * (BN - live); e += nw * 32) {
        const int kb = e / (BN - live), r = live + e % (BN - live);
        if (!bounds_ok(kb < KB && r < BN && kb * BN + r < slot_stride)) continue;
        sa_slots[kb * BN + r] = 0.f;
        sa_slots[slot_stride + kb * BN + r] = 0.f;
    }
}

template <int BN>
__device__ __forceinline__ void quantize_activations(const Params& p, uint8_t* a_res, float* sa_slots,
                                                     int slot_stride, int qw, int nw, int lane) {
    constexpr int kU = 4;                       // units in flight per warp
    const int KB = p.KB;
    const int live = p.M < 8 ? p.M : 8;         // the dispatch bound: at most 8 rows
    zero_rows<BN>(KB, live, a_res, sa_slots, slot_stride, qw, nw, lane);
    const int slots = (KB + 1) / 2;
    const int units = live * slots;
    const int h = lane >> 4;                    // half-warp h of slot i holds group 2i + h
    const int c16 = (lane & 15) >> 1;           // 16-byte chunk of the lane's 8 codes in the group's row
    for (int u0 = qw; u0 < units; u0 += kU * nw) {
        uint4 raw[kU];
        int row[kU], kb[kU];
        bool on[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int u = u0 + j * nw;
            row[j] = u / slots;
            const int slot = u - row[j] * slots;
            kb[j] = 2 * slot + h;
            on[j] = u < units && kb[j] < KB;    // odd KB: the last slot's second half is past the row
            raw[j] = make_uint4(0, 0, 0, 0);
            if (on[j] && bounds_ok(row[j] < p.M && (slot * 32 + lane) * 8 + 8 <= p.K))
                raw[j] = __ldg(reinterpret_cast<const uint4*>(p.a_bf16 + static_cast<int64_t>(row[j]) * p.lda_bf16 +
                                                               (slot * 32 + lane) * 8));
        }
        float2 x[kU][4];
        float amax[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            unpack8(raw[j], x[j]);
            amax[j] = fmaxf(fmaxf(fmaxf(fabsf(x[j][0].x), fabsf(x[j][0].y)), fmaxf(fabsf(x[j][1].x), fabsf(x[j][1].y))),
                            fmaxf(fmaxf(fabsf(x[j][2].x), fabsf(x[j][2].y)), fmaxf(fabsf(x[j][3].x), fabsf(x[j][3].y))));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
            for (int j = 0; j < kU; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            if (!on[j]) continue;
            const GroupQuant gq = make_group_quant(amax[j]);
            bool ok;
            uint2 codes = quant8_bracket(x[j], gq, ok);
            if (!ok) codes = quant8_divide(x[j], gq.scale);
            const int r = row[j];
            if (!bounds_ok(r < 8 && kb[j] < KB && kb[j] * BN + r < slot_stride)) continue;
            *reinterpret_cast<uint2*>(a_res + kb[j] * (8 * kBK) + r * kBK + ((c16 ^ (r & 7)) << 4) + (lane & 1) * 8) =
                codes;
            if ((lane & 15) == 0) {
                sa_slots[kb[j] * BN + r] = gq.scale;
                sa_slots[slot_stride + kb[j] * BN + r] = gq.scale;
            }
        }
    }
}

// In-kernel RMSNorm + per-1x128 quantization of the decode rows (the fused
// norm+quant of the q latent, then the GEMM, in one launch).  The live rows
// are cut into 256-column units (one row slot: a group per half-warp) spread
// over the nw quantizer warps, four per warp, as in quantize_activations, so
// that one row's loads and arithmetic run on several warps at once:
//   1. each warp loads its units' row chunks, sums the squares of each unit
//      across the warp and leaves the sum in shared memory;
//   2. after a barrier of the quantizer warps, each warp adds its row's unit
//      sums in slot order, takes r = 1/sqrt(ssq/K + eps) with IEEE
//      operations, reads the chunk again (from L1) with gamma, forms
//      x^ = (x r) gamma and quantizes its units.
// (The fp32 summation order differs from the norm+quant kernel's; both are
// checked against the oracle.)  The dispatch bound (M * slots <= 40) keeps
// every unit in one round of four per warp over the ten quantizer warps.
template <int BN>
__device__ __forceinline__ void norm_quantize_activations(const Params& p, uint8_t* a_res, float* sa_slots,
                                                          int slot_stride, int qw, int nw, int lane) {
    constexpr int kU = 4;                       // units per warp
    constexpr int kMaxSlots = 8;                // 256 columns per slot: K <= 2048
    __shared__ float unit_ssq[16 * kMaxSlots];  // [row][slot], rows < 16 (MMA N = 16)
    const int KB = p.KB;
    const int live = p.M < 8 ? p.M : 8;         // the dispatch bound: at most 8 rows
    zero_rows<BN>(KB, live, a_res, sa_slots, slot_stride, qw, nw, lane);
    const int slots = (KB + 1) / 2;
    const int units = live * slots;
    const int h = lane >> 4;                    // half-warp h of slot i holds group 2i + h
    const int c16 = (lane & 15) >> 1;
    const bool side = blockIdx.x == 0;
    const int K = KB * kBK;
    if (!bounds_ok(units <= kU * nw && slots <= kMaxSlots && p.M <= 8)) return;   // (debug build) outside the dispatch bound

    int row[kU] = {}, slot[kU] = {};
    bool on[kU] = {}, in[kU] = {};
    // The lane's chunk of unit j (odd KB: the last slot's second half is past
    // the row and reads as zero).
    auto load_unit = [&](int j) {
        return in[j] ? __ldg(reinterpret_cast<const uint4*>(p.a_bf16 + static_cast<int64_t>(row[j]) * p.lda_bf16 +
                                                             (slot[j] * 32 + lane) * 8))
                     : make_uint4(0, 0, 0, 0);
    };
    uint4 raw[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
        const int u = qw + j * nw;
        on[j] = u < units;
        row[j] = on[j] ? u / slots : 0;
        slot[j] = on[j] ? u - row[j] * slots : 0;
        in[j] = on[j] && (slot[j] * 32 + lane) * 8 + 8 <= K && bounds_ok(row[j] < p.M);
        raw[j] = load_unit(j);
    }
    // 1. The squares, summed per unit across the warp.
#pragma unroll
    for (int j = 0; j < kU; ++j) {
        float2 x[4];
        unpack8(raw[j], x);
        float2 sq = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) sq = fma2(x[t], x[t], sq);
        const float s = warp_sum(sq.x + sq.y);
        if (on[j] && lane == 0) unit_ssq[row[j] * kMaxSlots + slot[j]] = s;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nw * 32) : "memory");   // the quantizer warps only

#pragma unroll
    for (int j = 0; j < kU; ++j) {
        if (!on[j]) continue;
        float ssq = 0.f;
        for (int i = 0; i < slots; ++i) ssq += unit_ssq[row[j] * kMaxSlots + i];
        const float r = 1.0f / sqrtf(ssq / p.kq_f + p.eps);   // correctly rounded sqrt and divide
        const float2 r2 = make_float2(r, r);
        // The chunk again (an L1 hit: this warp read it above) and gamma.
        const uint4 graw = in[j] ? __ldg(reinterpret_cast<const uint4*>(p.gamma_q + (slot[j] * 32 + lane) * 8))
                                 : make_uint4(0, 0, 0, 0);
        float2 x[4], g[4];
        unpack8(load_unit(j), x);
        unpack8(graw, g);
#pragma unroll
        for (int t = 0; t < 4; ++t) x[t] = mul2(mul2(x[t], r2), g[t]);
        float amax = fmaxf(fmaxf(fmaxf(fabsf(x[0].x), fabsf(x[0].y)), fmaxf(fabsf(x[1].x), fabsf(x[1].y))),
                           fmaxf(fmaxf(fabsf(x[2].x), fabsf(x[2].y)), fmaxf(fabsf(x[3].x), fabsf(x[3].y))));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int m = row[j], kb = 2 * slot[j] + h;
        if (kb >= KB) continue;                 // odd KB: past the row (this half-warp only; no shuffles follow)
        if (!bounds_ok(m < 8 && m < p.M && kb * BN + m < slot_stride)) continue;
        const GroupQuant gq = make_group_quant(amax);
        bool ok;
        uint2 codes = quant8_bracket(x, gq, ok);
        if (!ok) codes = quant8_divide(x, gq.scale);
        *reinterpret_cast<uint2*>(a_res + kb * (8 * kBK) + m * kBK + ((c16 ^ (m & 7)) << 4) + (lane & 1) * 8) = codes;
        if ((lane & 15) == 0) {
            sa_slots[kb * BN + m] = gq.scale;
            sa_slots[slot_stride + kb * BN + m] = gq.scale;
        }
        if (side && p.q_out && bounds_ok((slot[j] * 32 + lane) * 8 + 8 <= K))
            *reinterpret_cast<uint2*>(p.q_out + static_cast<int64_t>(m) * K + (slot[j] * 32 + lane) * 8) = codes;
        if (side && p.qs_out && (lane & 15) == 0) p.qs_out[static_cast<int64_t>(kb) * p.M + m] = gq.scale;
    }
}

// The kv latent's rows of the fused call (CTA 0, after the q operand is
// ready: off the GEMM's path): RMSNorm as for the q rows above, bf16 out.
__device__ __forceinline__ void norm_kv_rows(const Params& p, int qw, int nw, int lane) {
    constexpr int kMaxSlots = 8;                // Kkv <= 2048
    const int kchunks = p.kkv / 8;
    for (int m = qw; m < p.M; m += nw) {
        const __nv_bfloat16* krow = p.kv + static_cast<int64_t>(m) * p.ldkv;
        uint4 raw[kMaxSlots], graw[kMaxSlots];
#pragma unroll
        for (int i = 0; i < kMaxSlots; ++i) {
            raw[i] = graw[i] = make_uint4(0, 0, 0, 0);
            if (i * 32 + lane < kchunks && bounds_ok(m < p.M)) {
                raw[i] = __ldg(reinterpret_cast<const uint4*>(krow + (i * 32 + lane) * 8));
                graw[i] = __ldg(reinterpret_cast<const uint4*>(p.gamma_kv + (i * 32 + lane) * 8));
            }
        }
        float2 skv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kMaxSlots; ++i) {
            if (i * 32 >= kchunks) break;
            float2 x[4];
            unpack8(raw[i], x);
#pragma unroll
            for (int t = 0; t < 4; ++t) skv[t & 1] = fma2(x[t], x[t], skv[t & 1]);
        }
        const float ssq_kv = warp_sum((skv[0].x + skv[1].x) + (skv[0].y + skv[1].y));
        const float rkv = 1.0f / sqrtf(ssq_kv / p.kkv_f + p.eps);
        const float2 rk2 = make_float2(rkv, rkv);
#pragma unroll
        for (int i = 0; i < kMaxSlots; ++i) {
            if (i * 32 + lane >= kchunks) continue;
            float2 x[4], g[4];
            unpack8(raw[i], x);
            unpack8(graw[i], g);
            uint4 v;
            __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 y = mul2(mul2(x[t], rk2), g[t]);
                hv[t] = __floats2bfloat162_rn(y.x, y.y);
            }
            if (bounds_ok(m < p.M && (i * 32 + lane) * 8 + 8 <= p.kkv))
                *reinterpret_cast<uint4*>(p.kv_out + static_cast<int64_t>(m) * p.ldkv_out + (i * 32 + lane) * 8) = v;
        }
    }
}

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

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS, int AQ = 0, int MINB = 1>
__global__ void __launch_bounds__(Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ>::kThreads, MINB)
block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_w0,
                         const __grid_constant__ CUtensorMap map_w1,
                         const __grid_constant__ CUtensorMap map_o0,
                         const __grid_constant__ CUtensorMap map_o1,
                         const Params p) {
    using C = Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled tiles.
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;
    uint8_t* a_res = smem + STAGES * C::kStageBytes;          // AQ: [KB + 1][8 rows][128] e4m3, resident
    uint8_t* out_stage = a_res + (AQ ? (p.KB + 1) * C::kResBytes : 0);   // [EPI_WARPS][kStageOutBytes]
    uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + EPI_WARPS * C::kStageOutBytes);
    uint64_t* full = bars;                    // [STAGES] TMA -> MMA
    uint64_t* empty = bars + STAGES;          // [STAGES] MMA -> TMA
    uint64_t* tfull = bars + 2 * STAGES;      // [NBUF]   MMA -> promotion
    uint64_t* tempty = tfull + NBUF;          // [NBUF]   promotion -> MMA
    uint64_t* sfull = tempty + NBUF;          // [2]      scale loader -> promotion
    uint64_t* sempty = sfull + 2;             // [2]      promotion -> scale loader
    uint64_t* drain = sempty + 2;             // [1]      abort drain of MMAs
    uint64_t* aready = drain + 1;             // [1]      AQ: quantizer warps -> MMA, promotion
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(aready + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // Scale slots (16-byte aligned), K blocks padded to KBP = a multiple of 4:
    // [2][KBP][kScaleCols] raw activation scales (per P row for non-swap, per
    // token for swap), then [2][KBP] weight scales.
    const int KBP = (p.KB + 3) & ~3;
    float* sa_slots = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_holder + 4) + 15) & ~uintptr_t(15));
    float* sw_slots = sa_slots + 2 * KBP * C::kScaleCols;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = p.total_tiles;
    const int KB = p.KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), EPI_WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sfull[i]), 32);            // one cp.async arrival per loader lane
            mbar_init(smem_u32(&sempty[i]), EPI_WARPS);
        }
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(aready), C::kThreads / 32 - 2);   // every warp but the producer and the MMA warp
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!AQ) tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_w0);
        tma_prefetch_desc(&map_w1);
        if (!SWAP) {
            tma_prefetch_desc(&map_o0);
            tma_prefetch_desc(&map_o1);
        }
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
    if (SWAP && warp == 0) {
        // Decode: the weight tiles of this CTA's first K blocks into L2 while
        // the previous kernel of the stream may still run (the weights are
        // the whole stream at decode sizes).  A prefetch only moves data into
        // L2, the point of coherence of global memory, so it cannot make a
        // later load read stale data even if an earlier kernel writes the
        // weights; the loads themselves still wait below.  (The same prefetch
        // in the 128 x 128 and CTA-pair kernels measured slower.)
        const int cap = kPrefetchKBlocks;
        int done = 0;
        for (int t = blockIdx.x; t < total && done < cap; t += gridDim.x, done += KB) {
            int pi, m0, n0;
            tile_coords<BN, SWAP>(p, t, pi, m0, n0);
            for (int kb = lane; kb < KB && done + kb < cap; kb += 32)
                tma_prefetch_l2(pi ? &map_w1 : &map_w0, kb * kBK, n0);
        }
    }
    // The producer's first tile, worked out before the dependency wait (it
    // reads only the launch parameters).
    int pre_pi = 0, pre_m0 = 0, pre_n0 = 0;
    if (warp == 0 && static_cast<int>(blockIdx.x) < total) tile_coords<BN, SWAP>(p, blockIdx.x, pre_pi, pre_m0, pre_n0);
    // Everything above reads no argument buffer; from here on every role
    // reads inputs (or writes outputs that an earlier kernel may still read).
    grid_dependency_wait();
    allow_dependent_launch();
    bounds_self_test(p.inject);

    if (AQ && warp >= 2) {
        // Quantize the activations once for all of this CTA's tiles, while the
        // producer already streams weights into the ring.
        if (AQ == 1)
            quantize_activations<BN>(p, a_res, sa_slots, KBP * C::kScaleCols, warp - 2, C::kThreads / 32 - 2, lane);
        else
            norm_quantize_activations<BN>(p, a_res, sa_slots, KBP * C::kScaleCols, warp - 2, C::kThreads / 32 - 2,
                                          lane);
        fence_proxy_async_smem();             // generic-proxy writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(aready));
        if (AQ == 2 && blockIdx.x == 0) norm_kv_rows(p, warp - 2, C::kThreads / 32 - 2, lane);
    }

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (2*STAGES lanes)
        // A thread's bulk copies complete one after another (about one per L2
        // round trip, measured on GB300), so every stage has its own pair of
        // lanes, each running its own loop: lane 2s loads the P tile of the K
        // blocks that use stage s (and arms the stage's barrier), lane 2s+1
        // their Q tile.  The lanes never wait for one another.
        if (lane < 2 * STAGES && !(AQ && (lane & 1))) {   // AQ: no activation copies
            const int ntl = blockIdx.x < total ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
            const uint32_t ng = static_cast<uint32_t>(ntl) * KB;   // K blocks of this CTA
            const int s = lane >> 1;
            const bool loads_q = lane & 1;
            const uint32_t fb = smem_u32(&full[s]);
            uint8_t* st = tiles + s * C::kStageBytes;
            uint32_t last = 0;     // 1 + the last K block this lane issued (0: none)
            bool ok = true;
            // The lanes wait on different barriers and so run apart: the (tile,
            // K block) position advances incrementally and the tile's
            // coordinates are recomputed only when the tile changes.
            int tl = s / KB, kbn = s % KB, cur_tl = -1;
            int pi = 0, m0 = 0, n0 = 0;
            for (uint32_t g = s; g < ng; g += STAGES) {
                // (The ring's first pass needs no wait: every stage starts free.)
                if (g >= STAGES && !wait_bounded(smem_u32(&empty[s]), ((g / STAGES) & 1) ^ 1, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                if (tl != cur_tl) {
                    if (tl == 0) {
                        pi = pre_pi;
                        m0 = pre_m0;
                        n0 = pre_n0;
                    } else {
                        tile_coords<BN, SWAP>(p, blockIdx.x + tl * gridDim.x, pi, m0, n0);
                    }
                    cur_tl = tl;
                }
                const int kb = kbn;
                kbn += STAGES;
                while (kbn >= KB) {
                    kbn -= KB;
                    ++tl;
                }
                if ((p.inject & 1u) && g == 0) continue;   // test hook: never arrive on full[0]
                const CUtensorMap* map_w = pi ? &map_w1 : &map_w0;
                if (!loads_q) {
                    mbar_arrive_expect_tx(fb, C::kStageBytes);
                    tma_load_2d(smem_u32(st), SWAP ? map_w : &map_a, fb, kb * kBK, SWAP ? n0 : m0);
                } else {
                    tma_load_2d(smem_u32(st + C::kPBytes), SWAP ? &map_a : map_w, fb, kb * kBK, SWAP ? m0 : n0);
                }
                last = g + 1;
            }
            if ((!ok || *abort_flag) && last > 0) {
                // Let this lane's last copy land before the CTA exits.
                const uint32_t g = last - 1;
                wait_drain(fb, (g / STAGES) & 1, tmo);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (whole warp, elected lane)
        constexpr uint32_t idesc = idesc_e4m3(BN);
        {
            // Descriptors of stage 0; stage s and K slice k only move the start
            // address field (16-byte units), which stays below 2^14 for 227 KB.
            const uint64_t dp0 = smem_desc_k_sw128(smem_u32(tiles));
            const uint64_t dq0 = smem_desc_k_sw128(smem_u32(AQ ? a_res : tiles + C::kPBytes));
            uint32_t g = 0;
            // Spinning waits (as on the MMA <-> promotion ring): a sleeping
            // wait here would add its wake-up latency to every launch.
            bool ok = !AQ || wait_bounded<true>(smem_u32(aready), 0, abort_flag, tmo), any = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int s = g % STAGES;
                    const int b = g % NBUF;
                    if (!wait_bounded<true>(smem_u32(&full[s]), (g / STAGES) & 1, abort_flag, tmo) ||
                        !wait_bounded<true>(smem_u32(&tempty[b]), ((g / NBUF) & 1) ^ 1, abort_flag, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                    // Q: the stage's slot, or the resident operand's K block.
                    const uint64_t qo = AQ ? static_cast<uint64_t>((kb * C::kResBytes) >> 4) : so;
                    const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        const uint64_t ko = static_cast<uint64_t>((k * kUmmaK) >> 4);
                        tc_mma_f8(d, dp0 + so + ko, dq0 + qo + ko, idesc, k > 0 ? 1u : 0u);
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
    } else if (warp == 3) {
        // ------------------------------------------------ scale loader (whole warp)
        // Raw activation scales of every K block of the CTA's next tile (per P
        // row, or per token for swap) and the tile's weight-scale row, copied
        // with cp.async into one of two shared slots; the slot's barrier
        // completes when every lane's copies have landed.
        int i = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
            const int slot = i & 1;
            const bool got = wait_bounded(smem_u32(&sempty[slot]), ((i >> 1) & 1) ^ 1, abort_flag, tmo);
            if (!__all_sync(0xffffffffu, got)) break;
            int pi, m0, n0;
            tile_coords<BN, SWAP>(p, t, pi, m0, n0);
            const Problem pr = pi ? p.prob[1] : p.prob[0];
            const float* sw = pr.w_scale + static_cast<int64_t>(n0 / kPRows) * pr.ld_ws;
            float* sa_dst = sa_slots + slot * KBP * C::kScaleCols;   // [kb][kScaleCols]
            const int rows = p.M - m0 < C::kScaleCols ? p.M - m0 : C::kScaleCols;
            if (AQ) {
                // Activation scales were written by the quantizer warps.
            } else if (p.vec_scales && rows == C::kScaleCols) {
                // Column-major scales with 16-byte aligned columns: each K block's
                // run of kScaleCols scales is contiguous, 16 bytes per lane per copy
                // (few, large copies: a thread's copies complete one at a time).
                constexpr int kVec = C::kScaleCols / 4;
                for (int e = lane; e < KB * kVec; e += 32) {
                    const int kb = e / kVec, v = e % kVec;
                    if (!bounds_ok(m0 + 4 * v + 4 <= p.M && kb * C::kScaleCols + 4 * v + 4 <= KBP * C::kScaleCols)) continue;
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sa_dst + kb * C::kScaleCols + 4 * v)),
                                 "l"(p.a_scale + static_cast<int64_t>(kb) * p.as_gs + m0 + 4 * v)
                                 : "memory");
                }
            } else {
                for (int e = lane; e < KB * C::kScaleCols; e += 32) {
                    const int kb = e / C::kScaleCols, j = e % C::kScaleCols;   // lanes walk rows: coalesced reads
                    const int m = m0 + j;
                    const bool live = m < p.M;                 // zero fill past the last row
                    const float* src = live ? p.a_scale + static_cast<int64_t>(m) * p.as_rs + kb * p.as_gs : p.a_scale;
                    if (!bounds_ok(e < KBP * C::kScaleCols)) continue;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(sa_dst + e)), "l"(src),
                                 "r"(live ? 4 : 0)
                                 : "memory");
                }
            }
            if (!bounds_ok(n0 / kPRows < (pr.N + kPRows - 1) / kPRows)) break;
            for (int kb = lane; kb < KB; kb += 32)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sw_slots + slot * KBP + kb)),
                             "l"(sw + kb)
                             : "memory");
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&sfull[slot]))
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy outlives the CTA
    } else if (warp >= 4) {
        // ------------------------------------------------ promotion + store
        const int ew = warp - 4;                 // 0 .. EPI_WARPS-1
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int slice = ew >> 2;               // column slice of the tile
        const int row = quarter * 32 + lane;     // P row (TMEM lane)
        const int col0 = slice * C::kCols;
        uint32_t g = 0;
        bool ok = true;
        if (AQ) ok = __all_sync(0xffffffffu, wait_bounded<true>(smem_u32(aready), 0, abort_flag, tmo));   // scales written
        int i = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
            int pi, m0, n0;
            tile_coords<BN, SWAP>(p, t, pi, m0, n0);
            const Problem pr = pi ? p.prob[1] : p.prob[0];
            const int slot = i & 1;
            {
                const bool got = wait_bounded(smem_u32(&sfull[slot]), (i >> 1) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) break;
            }
            const float* sa_t = sa_slots + slot * KBP * C::kScaleCols + (SWAP ? col0 : row);
            const float* sw_t = sw_slots + slot * KBP;

            float2 acc[C::kCols / 2];
#pragma unroll
            for (int j = 0; j < C::kCols / 2; ++j) acc[j] = make_float2(0.f, 0.f);

            // One K block: wait for its partial sum, read it out of TMEM, hand
            // the buffer back, and add it in with the per-column scales sc[j]
            // (pairs).  No shared-memory access here beyond the barriers: the
            // scales arrive in registers, fetched ahead of use, because shared
            // loads are slow while the tensor core streams its operands.
            auto promote = [&](const float2* sc, bool uniform) -> bool {
                const int b = g % NBUF;
                if (!bounds_ok(b * BN + col0 + C::kCols <= C::kTmemCols)) return false;
                // Every lane polls (each acquires the phase); the outcome is made
                // warp-uniform before the warp-collective TMEM load.
                const bool got = wait_bounded<true>(smem_u32(&tfull[b]), (g / NBUF) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) return false;
                tc_fence_after();
                uint64_t r[C::kCols / 2];
                tmem_ld_pairs<C::kCols>(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                            static_cast<uint32_t>(b * BN + col0),
                                        r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty[b]));
#pragma unroll
                for (int j = 0; j < C::kCols / 2; ++j)
                    acc[j] = __ffma2_rn(as_float2(r[j]), uniform ? sc[0] : sc[j], acc[j]);
                ++g;
                return true;
            };

            if (!SWAP) {
                // Four K blocks of scales per 16-byte load, the next four fetched
                // while the current four are promoted.
                auto sa4 = [&](int c) {   // this row's scales of K blocks c..c+3 (slot is [kb][row])
                    return make_float4(sa_t[(c + 0) * kPRows], sa_t[(c + 1) * kPRows], sa_t[(c + 2) * kPRows],
                                       sa_t[(c + 3) * kPRows]);
                };
                float4 a_cur = sa4(0);
                float4 w_cur = *reinterpret_cast<const float4*>(sw_t);
                for (int c = 0; c < KB && ok; c += 4) {
                    float4 a_nxt = a_cur, w_nxt = w_cur;
                    if (c + 4 < KB) {
                        a_nxt = sa4(c + 4);
                        w_nxt = *reinterpret_cast<const float4*>(sw_t + c + 4);
                    }
                    const float sk[4] = {a_cur.x * w_cur.x, a_cur.y * w_cur.y, a_cur.z * w_cur.z, a_cur.w * w_cur.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (c + u >= KB) break;
                        const float2 s2 = make_float2(sk[u], sk[u]);
                        if (!promote(&s2, true)) {
                            ok = false;
                            break;
                        }
                    }
                    a_cur = a_nxt;
                    w_cur = w_nxt;
                }
            } else {
                // The thread's kCols token scales of the next K block are fetched
                // while the current one is promoted.
                float4 a_cur[C::kScaleRegs], a_nxt[C::kScaleRegs];
                float w_cur = sw_t[0], w_nxt = w_cur;
#pragma unroll
                for (int q = 0; q < C::kScaleRegs; ++q) a_cur[q] = reinterpret_cast<const float4*>(sa_t)[q];
                for (int kb = 0; kb < KB; ++kb) {
                    if (kb + 1 < KB) {
                        const float* nx = sa_t + (kb + 1) * C::kScaleCols;
#pragma unroll
                        for (int q = 0; q < C::kScaleRegs; ++q) a_nxt[q] = reinterpret_cast<const float4*>(nx)[q];
                        w_nxt = sw_t[kb + 1];
                    }
                    float2 sc[C::kCols / 2];
                    const float2 w2 = make_float2(w_cur, w_cur);
#pragma unroll
                    for (int q = 0; q < C::kScaleRegs; ++q) {
                        sc[2 * q] = __fmul2_rn(make_float2(a_cur[q].x, a_cur[q].y), w2);
                        sc[2 * q + 1] = __fmul2_rn(make_float2(a_cur[q].z, a_cur[q].w), w2);
                    }
                    if (!promote(sc, false)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int q = 0; q < C::kScaleRegs; ++q) a_cur[q] = a_nxt[q];
                    w_cur = w_nxt;
                }
            }
            if (!ok) break;
            // This tile's scales are no longer read.
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sempty[slot]));

            if (!SWAP) {
                // bf16 block of this warp -> shared (64-byte swizzle: 16-byte
                // chunk c of row r sits at chunk c ^ ((r >> 1) & 3)) -> one TMA store.
                uint8_t* stg = out_stage + ew * C::kStageOutBytes;
                if (lane == 0) bulk_wait_read_all();   // the previous tile's store has read the buffer
                __syncwarp();
#pragma unroll
                for (int c = 0; c < C::kCols / 8; ++c) {
                    uint4 v;
                    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(acc[4 * c + q].x, acc[4 * c + q].y);
                    const int sc = c ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4*>(stg + lane * (C::kCols * 2) + sc * 16) = v;
                }
                fence_proxy_async_smem();              // generic-proxy writes -> visible to TMA
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(pi ? &map_o1 : &map_o0, smem_u32(stg), n0 + col0, m0 + quarter * 32);
                    bulk_commit();
                }
            } else {
                const int n = n0 + row;
                if (n < pr.N) {
#pragma unroll
                    for (int j = 0; j < C::kCols; ++j) {
                        const int m = m0 + col0 + j;
                        const float v = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
                        if (m < p.M && bounds_ok(m >= 0 && n >= 0 && n < pr.N))
                            pr.out[static_cast<int64_t>(m) * pr.ldo + n] = __float2bfloat16_rn(v);
                    }
                }
            }
        }
    }

    if (!SWAP && warp >= 4 && lane == 0) bulk_wait_all();   // stores complete before the CTA exits
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::kTmemCols)
                     : "memory");
    }
}

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS, int AQ = 0>
constexpr size_t smem_bytes(int KB) {
    using C = Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ>;
    const int KBP = (KB + 3) & ~3;
    return 1024 /* alignment slack */ + STAGES * C::kStageBytes + (AQ ? static_cast<size_t>(KB + 1) * C::kResBytes : 0) +
           EPI_WARPS * C::kStageOutBytes + (2 * STAGES + 2 * NBUF + 6) * 8 + 16 + 16 +
           static_cast<size_t>(2 * KBP * C::kScaleCols + 2 * KBP) * 4;
}

// ------------------------------------------------------------ CTA-pair kernel
//
// Large M.  A cluster of two CTAs on two SMs computes a 256 x 256 output tile
// with tcgen05.mma.cta_group::2 (MMA shape M=256, N=256).  CTA r (cluster
// rank r) holds activation rows 128r..128r+127 and weight rows 128r..128r+127
// of the tile in its own shared memory; the even CTA issues the MMAs, which
// read both CTAs' operands and leave each CTA's 128 x 256 fp32 partial sum in
// that CTA's TMEM.  Per SM and K block this lands 32 KB of operands for twice
// the MMA work of a 128 x 128 tile: on GB300 one SM takes in about 80-115 B
// per clock from L2 under load (measured), less than the 128 B/clock that
// 128 x 128 tiles need at the full MMA rate, and more than the 64 B/clock
// these tiles need.
//
// Roles as in block_scaled_gemm_kernel; the MMA warp runs in the even CTA
// only.  Both CTAs' loads signal the even CTA's stage barrier
// (TMA .cta_group::2); the MMA completions are multicast to both CTAs'
// "stage free" and "partial ready" barriers; both CTAs' promotion warps
// release a TMEM buffer on the even CTA's barrier.
//
// A K block is four MMAs of the whole tile (M=256, N=256, K=32: 128 cycles
// of tensor work per SM each) into one of two TMEM buffers of 256 columns;
// each CTA supplies half of the MMA's N, CTA r storing weight rows
// 128r .. 128r+127 of the tile.  Measured on GB300, an MMA of N=128 (64
// cycles of work) cannot be issued faster than ~87 cycles even back to back,
// while N=256 MMAs run at the full rate with waits in between; N=256 also
// reads the A tile once per K slice (32 KB of shared-memory reads per K block
// and SM, against the 32 KB the TMA writes).
//
// With only two buffers, the MMAs of K block g+2 wait for the promotion of
// K block g, so promotion must read a 256-column buffer out of TMEM quickly.
// Eight promotion warps (two per TMEM lane quarter, 128 columns each) hold
// 128 fp32 accumulators plus a 64-column TMEM load per thread (the compiler
// allocates the launch's 168 registers per thread; setmaxnreg moves the role
// warps' share to the promotion warps at run time).  Warp 2 issues the output
// stores, so that a promotion warp's epilogue is only its conversion and
// shared-memory writes: with the stores issued by the promotion warps
// themselves (they wait behind the operand loads in the TMA queue) the kernel
// took 330 instead of 308 us at M=8192.
namespace pair {
constexpr int kBN = 256;                        // output columns of a tile (both CTAs), the MMA's N
constexpr int kHalfN = 128;                     // weight rows each CTA supplies (half of the MMA's N)
constexpr int kStages = 4;
constexpr int kNBuf = 2;                        // K blocks in TMEM (256 columns each)
constexpr int kEpiWarps = 8;                    // two per TMEM lane quarter
constexpr int kThreads = (4 + kEpiWarps) * 32;
constexpr int kHalfBytes = kPRows * kBK;        // 16 KB: 128 rows x 128 K bytes
constexpr int kStageBytes = 2 * kHalfBytes;     // this CTA's activation rows + weight rows
constexpr int kCols = kBN / (kEpiWarps / 4);    // accumulator columns per promotion thread (128)
constexpr int kLdCols = 64;                     // columns per TMEM load
constexpr int kOutBlock = 64;                   // columns per output store box (128-byte rows)
constexpr int kStageOutBytes = 32 * kCols * 2;  // a promotion warp's 32 x 128 bf16 block
constexpr int kTmemCols = 512;
constexpr uint32_t kRegsLaunch = 168;           // 65536 / 384, in steps of 8
constexpr uint32_t kRegsRole = 40;
constexpr uint32_t kRegsEpi = 232;
static_assert(4 * 32 * kRegsRole + kEpiWarps * 32 * kRegsEpi <= kThreads * kRegsLaunch,
              "the register split must fit in what the block is launched with");
static_assert(kNBuf * kBN <= kTmemCols, "TMEM holds 512 fp32 columns");
static_assert(kCols % kLdCols == 0 && kCols % kOutBlock == 0, "whole loads and store boxes per thread");

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// All threads of both CTAs arrive, then wait for all.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrival on a barrier of the peer CTA.  Relaxed: the only thing it reports
// is that this warp's TMEM loads have completed (tcgen05.wait::ld), which
// needs no release of earlier memory operations; a release at cluster scope
// measured ~1000 cycles per arrival on GB300.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Tiled load into this CTA's shared memory whose completion is counted on a
// barrier of this CTA or of its peer (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the barrier at offset `bar` of both CTAs once the MMAs issued so
// far have completed.
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
        ::"r"(bar), "h"(static_cast<uint16_t>(0x3))
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
// Instruction descriptor: D fp32, A and B E4M3, K-major, M = 256, N = 256.
__host__ __device__ constexpr uint32_t idesc_e4m3_pair() {
    return (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
}

constexpr size_t smem_bytes(int KB) {
    const int KBP = (KB + 3) & ~3;
    return 1024 + kStages * kStageBytes + kEpiWarps * kStageOutBytes + (2 * kStages + 2 * kNBuf + 7) * 8 + 32 +
           static_cast<size_t>(2 * KBP * kPRows + 2 * 2 * KBP) * 4;
}
}  // namespace pair

__global__ void __launch_bounds__(pair::kThreads, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w0,
                 const __grid_constant__ CUtensorMap map_w1, const __grid_constant__ CUtensorMap map_o0,
                 const __grid_constant__ CUtensorMap map_o1, const Params p) {
    using namespace pair;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;
    uint8_t* out_stage = smem + kStages * kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + kEpiWarps * kStageOutBytes);
    uint64_t* full = bars;                    // [S]  even CTA: both CTAs' loads of a stage
    uint64_t* empty = bars + kStages;         // [S]  MMA -> TMA (multicast to both)
    uint64_t* tfull = bars + 2 * kStages;     // [NB] MMA -> promotion (multicast to both)
    uint64_t* tempty = tfull + kNBuf;         // [NB] even CTA: both CTAs' promotion -> MMA
    uint64_t* sfull = tempty + kNBuf;         // [2]
    uint64_t* sempty = sfull + 2;             // [2]
    uint64_t* drain = sempty + 2;             // [1]
    uint64_t* ofull = drain + 1;              // [1]  promotion warps -> store warp: staging written
    uint64_t* ofree = ofull + 1;              // [1]  store warp -> promotion warps: staging read by the stores
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(ofree + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int KBP = (p.KB + 3) & ~3;
    float* sa_slots = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_holder + 8) + 15) & ~uintptr_t(15));
    float* sw_slots = sa_slots + 2 * KBP * kPRows;     // [2][2 blocks][KBP]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool even = rank == 0;
    const int first = static_cast<int>(cluster_id_x()), stride = static_cast<int>(cluster_count_x());
    const int items = first < p.total_super ? (p.total_super - 1 - first) / stride + 1 : 0;
    const int KB = p.KB;

    // Tile t -> problem, first activation row of this CTA, first output column.
    auto coords = [&](int t, int& pi, int& m0, int& n0) {
        pi = t < p.super0 ? 0 : 1;
        if (pi) t -= p.super0;
        m0 = (t % p.tiles_m2) * 256 + static_cast<int>(rank) * kPRows;
        n0 = (t / p.tiles_m2) * kBN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < kNBuf; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 2 * kEpiWarps);   // every promotion warp of both CTAs
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sfull[i]), 32);
            mbar_init(smem_u32(&sempty[i]), kEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(ofull), kEpiWarps);
        mbar_init(smem_u32(ofree), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_w0);
        tma_prefetch_desc(&map_w1);
        tma_prefetch_desc(&map_o0);
        tma_prefetch_desc(&map_o1);
    }
    if (warp == 1) {
        // One warp of each CTA of the pair allocates, collectively.
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // both CTAs' barriers exist before any load or arrival targets them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint64_t tmo = p.timeout_ns;
    grid_dependency_wait();      // as in block_scaled_gemm_kernel
    allow_dependent_launch();
    bounds_self_test(p.inject);

    // Warp-group 0 (the role warps) hands registers to the promotion warps.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRole));
    if (warp == 0) {
        // ------------------------------------------------ TMA producer (2*S lanes, both CTAs)
        if (lane < 2 * kStages) {
            const uint32_t ng = static_cast<uint32_t>(items) * KB;
            const int s = lane >> 1;
            const int part = lane & 1;           // 0: activation rows, 1: weight rows
            const uint32_t fb = peer_addr(smem_u32(&full[s]), 0);   // the even CTA's stage barrier
            uint8_t* st = tiles + s * kStageBytes;
            uint32_t last = 0;
            bool ok = true;
            // The lanes of this warp wait on different barriers, so they run
            // apart and each executes its own instructions: the (tile, K
            // block) position advances incrementally and the tile's
            // coordinates are recomputed only when the tile changes.
            int tl = s / KB, kb = s % KB, cur_tl = -1;
            int pi = 0, m0 = 0, n0 = 0;
            for (uint32_t g = s; g < ng; g += kStages) {
                if (!wait_bounded(smem_u32(&empty[s]), ((g / kStages) & 1) ^ 1, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                if (tl != cur_tl) {
                    coords(first + tl * stride, pi, m0, n0);
                    cur_tl = tl;
                }
                const int kbi = kb;
                kb += kStages;
                while (kb >= KB) {
                    kb -= KB;
                    ++tl;
                }
                if ((p.inject & 1u) && g == 0) continue;   // test hook: never arrive on full[0]
                if (part == 0) {
                    if (even) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * kStageBytes);
                    tma_load_2d_pair(smem_u32(st), &map_a, fb, kbi * kBK, m0);
                } else {
                    tma_load_2d_pair(smem_u32(st + kHalfBytes), pi ? &map_w1 : &map_w0, fb, kbi * kBK,
                                     n0 + static_cast<int>(rank) * kHalfN);
                }
                last = g + 1;
            }
            if (ok && last > 0) {
                // Tail: the stage is released once the MMAs have read this lane's
                // last copy, i.e. once the last arrival aimed at this CTA has landed.
                const uint32_t gn = last - 1 + kStages;
                ok = wait_bounded(smem_u32(&empty[s]), ((gn / kStages) & 1) ^ 1, abort_flag, tmo);
            }
            if ((!ok || *abort_flag) && last > 0) {
                // Abort: this lane's last copy may still be landing in this CTA's
                // shared memory.  Its completion is counted on the even CTA's
                // stage barrier, so the even CTA waits (bounded) for that phase;
                // the odd CTA cannot wait on a peer's barrier and lets a fixed,
                // generous settle time pass instead.  Both then meet at the
                // cluster barrier before either releases its memory.
                if (even) wait_drain(smem_u32(&full[s]), ((last - 1) / kStages) & 1, tmo);
                else settle_ns(kAbortSettleNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA, whole warp)
        if (even) {
            constexpr uint32_t idesc = idesc_e4m3_pair();
            const uint64_t da0 = smem_desc_k_sw128(smem_u32(tiles));
            const uint64_t dw0 = smem_desc_k_sw128(smem_u32(tiles + kHalfBytes));
            uint32_t g = 0;
            bool ok = true, any = false;
            for (int it = 0; it < items && ok; ++it) {
                for (int kb = 0; kb < KB && ok; ++kb, ++g) {
                    const int s = g % kStages;
                    const int q = g % kNBuf;
                    const uint64_t so = static_cast<uint64_t>((s * kStageBytes) >> 4);
                    if (!wait_bounded<true>(smem_u32(&full[s]), (g / kStages) & 1, abort_flag, tmo) ||
                        !wait_bounded<true>(smem_u32(&tempty[q]), ((g / kNBuf) & 1) ^ 1, abort_flag, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(q * kBN);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        const uint64_t ko = static_cast<uint64_t>((k * kUmmaK) >> 4);
                        tc_mma_f8_pair(d, da0 + so + ko, dw0 + so + ko, idesc, k > 0 ? 1u : 0u);
                    }
                    tc_commit_pair_both(smem_u32(&empty[s]));    // stage free once these MMAs have read it
                    tc_commit_pair_both(smem_u32(&tfull[q]));    // partial sum ready (both CTAs)
                    any = true;
                }
            }
            if (*abort_flag && any) {
                tc_commit_pair_local(smem_u32(drain));
                wait_drain(smem_u32(drain), 0, tmo);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ output stores (lane 0, both CTAs)
        // The promotion warps write a tile's bf16 blocks into their staging
        // buffers; this warp issues the TMA stores and hands the buffers back
        // once the stores have read them, so that issuing the stores (which
        // waits behind the operand loads in the TMA queue) stays off the
        // promotion warps' path.
        if (lane == 0) {
            for (int i = 0; i < items; ++i) {
                if (!wait_bounded(smem_u32(ofull), i & 1, abort_flag, tmo)) break;
                int pi, m0, n0;
                coords(first + i * stride, pi, m0, n0);
                const Problem pr = pi ? p.prob[1] : p.prob[0];
                for (int ew = 0; ew < kEpiWarps; ++ew) {
                    const int quarter = (ew + 4) & 3, col0 = (ew >> 2) * kCols;
                    if (m0 + quarter * 32 >= p.M || n0 + col0 >= pr.N) continue;
                    uint8_t* stg = out_stage + ew * kStageOutBytes;
                    for (int ob = 0; ob < kCols / kOutBlock; ++ob)
                        if (n0 + col0 + ob * kOutBlock < pr.N)
                            tma_store_2d(pi ? &map_o1 : &map_o0, smem_u32(stg + ob * (32 * kOutBlock * 2)),
                                         n0 + col0 + ob * kOutBlock, m0 + quarter * 32);
                }
                bulk_commit();
                bulk_wait_read_all();            // the stores have read the staging buffers
                mbar_arrive(smem_u32(ofree));
            }
            bulk_wait_all();                     // every store has completed before the CTA exits
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------ scale loader (whole warp, both CTAs)
        for (int i = 0; i < items; ++i) {
            const int slot = i & 1;
            const bool got = wait_bounded(smem_u32(&sempty[slot]), ((i >> 1) & 1) ^ 1, abort_flag, tmo);
            if (!__all_sync(0xffffffffu, got)) break;
            int pi, m0, n0;
            coords(first + i * stride, pi, m0, n0);
            const Problem pr = pi ? p.prob[1] : p.prob[0];
            float* sa_dst = sa_slots + slot * KBP * kPRows;     // [kb][128 rows]
            const int rows = p.M - m0;
            if (p.vec_scales && rows >= kPRows) {
                for (int e = lane; e < KB * (kPRows / 4); e += 32) {
                    const int kb = e / (kPRows / 4), v = e % (kPRows / 4);
                    if (!bounds_ok(m0 + 4 * v + 4 <= p.M && kb < KBP)) continue;
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sa_dst + kb * kPRows + 4 * v)),
                                 "l"(p.a_scale + static_cast<int64_t>(kb) * p.as_gs + m0 + 4 * v)
                                 : "memory");
                }
            } else {
                for (int e = lane; e < KB * kPRows; e += 32) {
                    const int kb = e / kPRows, j = e % kPRows;
                    const int m = m0 + j;
                    const bool live = m < p.M;
                    const float* src = live ? p.a_scale + static_cast<int64_t>(m) * p.as_rs + kb * p.as_gs : p.a_scale;
                    if (!bounds_ok(e < KBP * kPRows)) continue;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(sa_dst + e)), "l"(src),
                                 "r"(live ? 4 : 0)
                                 : "memory");
                }
            }
            // The tile's two 128-feature weight-scale blocks (a block past the
            // end, whose features are not stored, repeats the last one).
            const int nblocks = (pr.N + kPRows - 1) / kPRows;
            for (int e = lane; e < 2 * KB; e += 32) {
                const int h = e / KB, kb = e % KB;
                int nb = n0 / kPRows + h;
                nb = nb < nblocks ? nb : nblocks - 1;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sw_slots + (slot * 2 + h) * KBP + kb)),
                             "l"(pr.w_scale + static_cast<int64_t>(nb) * pr.ld_ws + kb)
                             : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&sfull[slot])) : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        // ------------------------------------------------ promotion + store (both CTAs)
        const int ew = warp - 4;
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int slice = ew >> 2;               // columns kCols*slice .. +kCols-1 of the tile
        const int row = quarter * 32 + lane;
        const int col0 = slice * kCols;
        static_assert(kNBuf == 2, "two buffer-free barriers in the even CTA");
        static_assert(kCols == kPRows, "a promotion thread's columns share one weight-scale block");
        const uint32_t tempty_even0 = peer_addr(smem_u32(&tempty[0]), 0);
        const uint32_t tempty_even1 = peer_addr(smem_u32(&tempty[1]), 0);
        uint32_t g = 0;
        bool ok = true;
        for (int i = 0; i < items && ok; ++i) {
            int pi, m0, n0;
            coords(first + i * stride, pi, m0, n0);
            const Problem pr = pi ? p.prob[1] : p.prob[0];
            const int slot = i & 1;
            {
                const bool got = wait_bounded(smem_u32(&sfull[slot]), (i >> 1) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) break;
            }
            const float* sa_t = sa_slots + slot * KBP * kPRows + row;
            const float* sw_t = sw_slots + (slot * 2 + slice) * KBP;

            float2 acc[kCols / 2];
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j) acc[j] = make_float2(0.f, 0.f);

            float a_nxt = sa_t[0], w_nxt = sw_t[0];
            for (int kb = 0; kb < KB; ++kb) {
                const float sk = a_nxt * w_nxt;
                if (kb + 1 < KB) {
                    a_nxt = sa_t[(kb + 1) * kPRows];
                    w_nxt = sw_t[kb + 1];
                }
                const int b = g % kNBuf;
                const bool got = wait_bounded<true>(smem_u32(&tfull[b]), (g / kNBuf) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float2 s2 = make_float2(sk, sk);
                if (!bounds_ok(b * kBN + col0 + kCols <= kTmemCols)) {
                    ok = false;
                    break;
                }
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(b * kBN + col0);
                // The thread's columns in 64-column loads, each added in before the
                // next is read; the buffer is released once the last load has
                // completed, before its columns are added.
#pragma unroll
                for (int c = 0; c < kCols / kLdCols; ++c) {
                    uint64_t r[kLdCols / 2];
                    tmem_ld_pairs<kLdCols>(tbase + c * kLdCols, r);
                    if (c == kCols / kLdCols - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (even)
                                mbar_arrive(smem_u32(&tempty[b]));
                            else
                                mbar_arrive_remote(b ? tempty_even1 : tempty_even0);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kLdCols / 2; ++j)
                        acc[c * (kLdCols / 2) + j] = __ffma2_rn(as_float2(r[j]), s2, acc[c * (kLdCols / 2) + j]);
                }
                ++g;
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sempty[slot]));

            // Epilogue: this warp's 32 rows x kCols columns as bf16 into its
            // staging buffer, as blocks of 64 columns (128-byte rows, 128-byte
            // swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)); warp 2
            // issues the TMA stores.  Every promotion warp signals every tile
            // (the store warp counts them), whether or not its block is in range.
            if (i > 0) {
                const bool got = wait_bounded(smem_u32(ofree), (i - 1) & 1, abort_flag, tmo);
                if (!__all_sync(0xffffffffu, got)) break;
            }
            if (m0 + quarter * 32 < p.M && n0 + col0 < pr.N) {
                uint8_t* stg = out_stage + ew * kStageOutBytes;
#pragma unroll
                for (int ob = 0; ob < kCols / kOutBlock; ++ob) {
#pragma unroll
                    for (int c = 0; c < kOutBlock / 8; ++c) {
                        uint4 v;
                        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = acc[ob * (kOutBlock / 2) + 4 * c + q];
                            hv[q] = __floats2bfloat162_rn(f.x, f.y);
                        }
                        *reinterpret_cast<uint4*>(stg + ob * (32 * kOutBlock * 2) + lane * (kOutBlock * 2) +
                                                  ((c ^ (lane & 7)) * 16)) = v;
                    }
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(ofull));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // no CTA leaves while its peer may still address its memory
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
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

// 2-D map over a bf16 output [rows, cols] with row stride ld elements; box =
// box_cols x 32 rows, box_cols = 32 (64-byte rows, 64-byte swizzle) or 64
// (128-byte rows, 128-byte swizzle), the staging layouts of the epilogues;
// stores past the extent are clipped.
bool make_out_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoding a tensor map is host work of a few microseconds, comparable to a
// decode-size GEMM, so maps are kept in a small cache.  A map only describes
// address arithmetic (base, extents, strides, box), so a cached map stays
// valid for its key whatever the memory holds.
struct MapKey {
    const void* base;
    int64_t rows, cols, ld;
    int box, kind;          // kind 0: operand map, 1: output map
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld && box == o.box && kind == o.kind;
    }
};

class MapCache {
  public:
    bool get(const MapKey& k, CUtensorMap* m) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSize; ++i)
            if (used_[i] && keys_[i] == k) {
                *m = maps_[i];
                return true;
            }
        return false;
    }
    void put(const MapKey& k, const CUtensorMap& m) {
        std::lock_guard<std::mutex> lock(mu_);
        keys_[next_] = k;
        maps_[next_] = m;
        used_[next_] = true;
        next_ = (next_ + 1) % kSize;
    }

  private:
    static constexpr int kSize = 64;
    std::mutex mu_;
    MapKey keys_[kSize] = {};
    CUtensorMap maps_[kSize] = {};
    bool used_[kSize] = {};
    int next_ = 0;
};

MapCache& map_cache() {
    static MapCache c;
    return c;
}

bool cached_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t ld, int box_rows) {
    const MapKey k{base, rows, K, ld, box_rows, 0};
    if (map_cache().get(k, m)) return true;
    if (!make_map(m, base, rows, K, ld, box_rows)) return false;
    map_cache().put(k, *m);
    return true;
}

bool cached_out_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols) {
    const MapKey k{base, rows, cols, ld, box_cols, 1};
    if (map_cache().get(k, m)) return true;
    if (!make_out_map(m, base, rows, cols, ld, box_cols)) return false;
    map_cache().put(k, *m);
    return true;
}

// cudaFuncSetAttribute once per (kernel, device, size): it is host work on
// every call otherwise.
bool set_smem_attr(const void* kern, size_t smem) {
    static std::mutex mu;
    static std::vector<std::tuple<const void*, int, size_t>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& d : done)
        if (std::get<0>(d) == kern && std::get<1>(d) == dev && std::get<2>(d) >= smem) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.emplace_back(kern, dev, smem);
    return true;
}

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

// Every CTA quantizes all M rows itself, so the in-GEMM quantization pays
// only while each of its ten quantizer warps has one batch of four 256-column
// units (measured on GB300 at K=1536, per call in a graph: M=1 11.1 us vs
// 13.1-13.4 us for the quant kernel then the GEMM, M=6 12.6 vs 13.1-13.4;
// with the bound raised, M=8 / 12 / 16 took 13.9 / 15.2 / 16.4 us against
// 13.1-13.4).  At most 8 rows (the resident operand's rows per K block),
// K <= 2048.
bool bf16a_in_gemm(int64_t M, int64_t K) {
    const int64_t slots = (K / 128 + 1) / 2;
    return M >= 1 && M <= 8 && K <= 2048 && M * slots <= 40;
}

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


// ---- Kernel variant of a call, chosen on the host from (M, K) alone.
// The variants and their shared-memory sizes per CTA (227 KB at most):
//   decode (M <= 64, swap-AB, tokens as the MMA's N = 16 / 32 / 64);
//   128 x 128 tiles (64 < M < 256; and M >= 256 when the CTA-pair kernel's
//     scale slots do not fit, K > 4096), five operand stages while they fit
//     beside the scale slots (K <= 4096), three beyond;
//   CTA pair, 256 x 256 tiles (M >= 256, K <= 4096);
//   decode on bf16 activations quantized (and normalized) in the prologue.
enum Variant : int32_t {
    kVarDecode16 = 1,
    kVarDecode32 = 2,
    kVarDecode64 = 3,
    kVarTile128 = 4,
    kVarTile128K = 5,          // three stages: room for the scale slots of long K
    kVarPair = 6,
    kVarDecodeQuant = 7,       // bf16 activations quantized in the prologue
    kVarDecodeNormQuant = 8,   // ... after an RMSNorm
};

constexpr size_t kMaxSmem = 227 * 1024;

size_t variant_smem(int v, int KB) {
    switch (v) {
        case kVarDecode16: return gemm::smem_bytes<16, true, 5, 16, 8>(KB);
        case kVarDecode32: return gemm::smem_bytes<32, true, 5, 8, 8>(KB);
        case kVarDecode64: return gemm::smem_bytes<64, true, 8, 8, 8>(KB);
        case kVarTile128: return gemm::smem_bytes<128, false, 5, 4, 16>(KB);
        case kVarTile128K: return gemm::smem_bytes<128, false, 3, 4, 16>(KB);
        case kVarPair: return gemm::pair::smem_bytes(KB);
        case kVarDecodeQuant: return gemm::smem_bytes<16, true, 6, 2, 8, 1>(KB);
        case kVarDecodeNormQuant: return gemm::smem_bytes<16, true, 5, 2, 8, 2>(KB);
    }
    return 0;
}

// aq: 0 pre-quantized activations, 1 bf16 quantized in the kernel, 2 the
// same after an RMSNorm.  UNSUPPORTED when no variant serves (M, K).
dsnq_status plan_gemm(int64_t M, int64_t K, int aq, int* variant, size_t* smem) {
    if (M < 1 || K < 128 || K % 128 != 0 || K > 8192 || M > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    const int KB = static_cast<int>(K / 128);
    int v;
    if (aq) {
        if (!bf16a_in_gemm(M, K)) return DSNQ_ERR_UNSUPPORTED;
        v = aq == 2 ? kVarDecodeNormQuant : kVarDecodeQuant;
    } else if (M <= 64) {
        v = M <= 16 ? kVarDecode16 : M <= 32 ? kVarDecode32 : kVarDecode64;
    } else if (M >= 256 && variant_smem(kVarPair, KB) <= kMaxSmem) {
        v = kVarPair;
    } else {
        v = variant_smem(kVarTile128, KB) <= kMaxSmem ? kVarTile128 : kVarTile128K;
    }
    const size_t bytes = variant_smem(v, KB);
    if (bytes > kMaxSmem) return DSNQ_ERR_UNSUPPORTED;
    *variant = v;
    *smem = bytes;
    return DSNQ_OK;
}

template <int BN, bool SWAP, int STAGES, int NBUF, int EPI_WARPS, int AQ = 0, int MINB = 1>
dsnq_status launch(gemm::Params& prm, const CUtensorMap& ma, const CUtensorMap& mw0, const CUtensorMap& mw1,
                   const CUtensorMap& mo0, const CUtensorMap& mo1, cudaStream_t stream) {
    using C = gemm::Cfg<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ>;
    auto kern = gemm::block_scaled_gemm_kernel<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ, MINB>;
    const size_t smem = gemm::smem_bytes<BN, SWAP, STAGES, NBUF, EPI_WARPS, AQ>(prm.KB);
    if (smem > 227 * 1024) return DSNQ_ERR_UNSUPPORTED;
    if (!set_smem_attr(reinterpret_cast<const void*>(kern), smem)) return DSNQ_ERR_CUDA;
    // Persistent: MINB CTAs per SM (as many as the shared-memory ring and
    // TMEM allow), each walking the tile space with a stride of the grid size.
    const int sms = device_sm_count() * MINB;
    const int grid = prm.total_tiles < sms ? prm.total_tiles : (sms > 0 ? sms : prm.total_tiles);
    return launch_result(launch_kernel(kern, dim3(grid), dim3(C::kThreads), smem, stream, ma, mw0, mw1, mo0, mo1, prm));
}

// CTA-pair kernel: as many 2-CTA clusters as fit at once, each walking the
// 256 x 256 tiles with a stride of the cluster count.
dsnq_status launch_pair(gemm::Params& prm, const CUtensorMap& ma, const CUtensorMap& mw0, const CUtensorMap& mw1,
                        const CUtensorMap& mo0, const CUtensorMap& mo1, cudaStream_t stream) {
    const size_t smem = gemm::pair::smem_bytes(prm.KB);
    if (smem > 227 * 1024) return DSNQ_ERR_UNSUPPORTED;
    auto kern = gemm::pair_gemm_kernel;
    if (!set_smem_attr(reinterpret_cast<const void*>(kern), smem)) return DSNQ_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(gemm::pair::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> fit{-1};     // clusters resident at once
    int clusters = fit.load();
    if (clusters < 0) {
        cfg.gridDim = dim3(2 * 128, 1, 1);
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return DSNQ_ERR_CUDA;
        }
        fit.store(clusters);
    }
    if (clusters <= 0) return DSNQ_ERR_UNSUPPORTED;
    const int n = prm.total_super < clusters ? prm.total_super : clusters;
    cfg.gridDim = dim3(2 * n, 1, 1);
    cfg.numAttrs = launch_overlap_enabled() ? 2 : 1;
    return launch_result(cudaLaunchKernelEx(&cfg, kern, ma, mw0, mw1, mo0, mo1, prm));
}

// The RMSNorm that precedes the in-kernel quantization, and its side
// outputs (validated by the caller).
struct NormSide {
    const void* gamma_q;
    const void* kv;
    int64_t ldkv;
    const void* gamma_kv;
    int64_t kkv;
    float eps;
    void* kv_out;
    int64_t ldkv_out;
    void* q_out;
    float* qs_out;
};

// a_bf16 != NULL selects the decode variant that quantizes bf16 activations
// itself (see bf16a_in_gemm), after an RMSNorm when ns != NULL; a, as and the
// scale layout are then unused.
dsnq_status run_gemm(int64_t M, int64_t K, const void* a, int64_t lda, const float* as,
                     dsnq_scale_layout layout, int64_t ld_as, const Consumer& c0, const Consumer& c1,
                     void* stream, const void* a_bf16 = nullptr, int64_t lda_bf16 = 0,
                     const NormSide* ns = nullptr) {
    const bool aq = a_bf16 != nullptr;
    if (M < 0 || K <= 0 || c0.N < 0 || c1.N < 0) return DSNQ_ERR_INVALID_ARG;
    if (!aq && layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0) return DSNQ_ERR_UNSUPPORTED;
    if (M > 0x7fffffffLL || K > 8192) return DSNQ_ERR_UNSUPPORTED;
    if (aq && !bf16a_in_gemm(M, K)) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;          // empty activations may come with NULL pointers
    const int64_t KB = K / 128;
    int64_t ld = 0;
    if (aq) {
        if (lda_bf16 < K) return DSNQ_ERR_INVALID_ARG;
        if (!aligned(a_bf16, 16) || lda_bf16 % 8) return DSNQ_ERR_MISALIGNED;
    } else {
        if (!a || !as) return DSNQ_ERR_INVALID_ARG;
        if (lda < K) return DSNQ_ERR_INVALID_ARG;
        ld = scale_ld(layout, M, KB, ld_as);
        if (ld < 0) return DSNQ_ERR_INVALID_ARG;
        if (!aligned(a, 16) || lda % 16 || !aligned(as, 4)) return DSNQ_ERR_MISALIGNED;
    }
    dsnq_status st = check_consumer(c0, K);
    if (st != DSNQ_OK) return st;
    st = check_consumer(c1, K);
    if (st != DSNQ_OK) return st;
    if (c0.N == 0 && c1.N == 0) return DSNQ_OK;

    // The variant: decode batches (M <= 64) run swap-AB, the tokens being the
    // MMA's N; from 256 rows on 256 x 256 tiles on CTA pairs; in between (and
    // for long K) 128 x 128 tiles with four TMEM partial buffers.
    int variant = 0;
    size_t smem_plan = 0;
    st = plan_gemm(M, K, aq ? (ns ? 2 : 1) : 0, &variant, &smem_plan);
    if (st != DSNQ_OK) return st;
    (void)smem_plan;
    const bool swap = variant <= kVarDecode64 || variant >= kVarDecodeQuant;
    const bool paired = variant == kVarPair;
    const int bn = swap ? (variant == kVarDecode32 ? 32 : variant == kVarDecode64 ? 64 : 16) : 128;
    const int a_box = swap ? bn : gemm::kPRows;
    // The CTA-pair kernel loads each CTA's 128 weight rows of a tile (its half
    // of the MMA's N=256) as one box.
    const int w_box = swap ? gemm::kPRows : (paired ? gemm::pair::kHalfN : bn);

    gemm::Params prm{};
    prm.M = static_cast<int>(M);
    prm.K = static_cast<int>(K);
    prm.KB = static_cast<int>(KB);
    prm.a_scale = as;
    if (layout == DSNQ_SCALE_ROW_MAJOR) { prm.as_rs = ld; prm.as_gs = 1; }
    else { prm.as_rs = 1; prm.as_gs = ld; }
    prm.vec_scales = !aq && layout == DSNQ_SCALE_COL_MAJOR && ld % 4 == 0 && aligned(as, 16);
    prm.a_bf16 = static_cast<const __nv_bfloat16*>(a_bf16);
    prm.lda_bf16 = lda_bf16;
    if (ns) {
        prm.gamma_q = static_cast<const __nv_bfloat16*>(ns->gamma_q);
        prm.kv = static_cast<const __nv_bfloat16*>(ns->kv);
        prm.ldkv = ns->ldkv;
        prm.gamma_kv = static_cast<const __nv_bfloat16*>(ns->gamma_kv);
        prm.kkv = static_cast<int>(ns->kkv);
        prm.kq_f = static_cast<float>(K);
        prm.kkv_f = static_cast<float>(ns->kkv);
        prm.eps = ns->eps;
        prm.kv_out = static_cast<__nv_bfloat16*>(ns->kv_out);
        prm.ldkv_out = ns->ldkv_out;
        prm.q_out = static_cast<uint8_t*>(ns->q_out);
        prm.qs_out = ns->qs_out;
    }
    const int64_t rows_per_a_tile = swap ? bn : gemm::kPRows;
    prm.tiles_m = static_cast<int>((M + rows_per_a_tile - 1) / rows_per_a_tile);

    CUtensorMap ma, mw[2], mo[2];
    if (!aq && !cached_map(&ma, a, M, K, lda, a_box)) return DSNQ_ERR_CUDA;
    const Consumer* cs[2] = {&c0, &c1};
    int64_t total = 0, total_super = 0;
    int np = 0;
    prm.tiles_m2 = static_cast<int>((M + 255) / 256);
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
        if (!cached_map(&mw[np], c.w, c.N, K, c.ldw, w_box)) return DSNQ_ERR_CUDA;
        if (!swap && !cached_out_map(&mo[np], c.out, M, c.N, c.ldo, paired ? 64 : 32)) return DSNQ_ERR_CUDA;
        const int64_t tiles = static_cast<int64_t>(prm.tiles_m) * pr.tiles_n;
        const int64_t supers = static_cast<int64_t>(prm.tiles_m2) * ((c.N + 255) / 256);
        if (np == 0) {
            prm.tiles0 = static_cast<int>(tiles);
            prm.super0 = static_cast<int>(supers);
        }
        total += tiles;
        total_super += supers;
        ++np;
    }
    if (np == 1) {
        mw[1] = mw[0];
        mo[1] = mo[0];
    }
    if (swap) mo[0] = mo[1] = mw[0];   // unused by the decode variant
    if (aq) ma = mw[0];                 // unused: the kernel quantizes the activations itself
    if (total > 0x7fffffffLL) return DSNQ_ERR_UNSUPPORTED;
    prm.total_tiles = static_cast<int>(total);
    prm.total_super = static_cast<int>(total_super);
    const uint64_t tmo = debug_wait_timeout_ns();
    prm.timeout_ns = tmo ? tmo : kDefaultTimeoutNs;
    prm.inject = debug_inject_flags();

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (variant) {
        // Decode on bf16 activations quantized (and normalized) in the
        // prologue: two CTAs per SM like the 16-token decode variant, so
        // that all 224 weight tiles stream in one wave (M=1: 14.1 -> 11.1 us
        // per call in a graph; with one CTA per SM, eight stages, 72 SMs
        // took a second tile).  The 8-row resident operand leaves room for
        // a sixth stage; two TMEM buffers suffice at these sizes.  Measured
        // per call in graphs of 100 at M=1 against five stages, sixteen
        // buffers and a 16-row operand: quantize only 10.33 -> 9.92-9.94 us,
        // norm+quant 11.17-11.19 -> 10.99-11.01 us (a sixth stage there:
        // 11.41 us).
        case kVarDecodeQuant: return launch<16, true, 6, 2, 8, 1, 2>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        case kVarDecodeNormQuant: return launch<16, true, 5, 2, 8, 2, 2>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        case kVarPair: return launch_pair(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        // Decode: the kernel streams the weights.  Up to 32 tokens two CTAs
        // share an SM (five stages, half of TMEM each), so that all 224
        // weight tiles of the DSv4 dual problem stream at once on 152 SMs
        // instead of 72 SMs taking a second tile after the others finish
        // (M=1: 12.1 -> 10.8 us per call in a graph).  The MMA per K block is
        // tiny, so the MMA <-> promotion round trip sets the pace within a
        // CTA; its TMEM ring (256 / BN buffers) lets the MMA run most of a
        // tile ahead of the promotion.  64 tokens keep one CTA per SM (two
        // measured 4x slower).
        case kVarDecode16: return launch<16, true, 5, 16, 8, 0, 2>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        case kVarDecode32: return launch<32, true, 5, 8, 8, 0, 2>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        case kVarDecode64: return launch<64, true, 8, 8, 8>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        case kVarTile128: return launch<128, false, 5, 4, 16>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
        default: return launch<128, false, 3, 4, 16>(prm, ma, mw[0], mw[1], mo[0], mo[1], s);
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

extern "C" dsnq_status dsnq_gemm_plan(int64_t M, int64_t K, int32_t* variant, int64_t* smem_bytes) {
    if (M < 0 || K <= 0) return DSNQ_ERR_INVALID_ARG;
    if (M == 0) {
        if (variant) *variant = 0;
        if (smem_bytes) *smem_bytes = 0;
        return DSNQ_OK;
    }
    int v = 0;
    size_t smem = 0;
    const dsnq_status st = plan_gemm(M, K, 0, &v, &smem);
    if (st != DSNQ_OK) return st;
    if (variant) *variant = v;
    if (smem_bytes) *smem_bytes = static_cast<int64_t>(smem);
    return DSNQ_OK;
}

extern "C" dsnq_status dsnq_bf16a_workspace_bytes(int64_t M, int64_t K, int64_t* code_bytes, int64_t* scale_bytes) {
    if (M < 0 || K <= 0) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > 4096) return DSNQ_ERR_UNSUPPORTED;
    const bool none = M == 0 || bf16a_in_gemm(M, K);
    if (code_bytes) *code_bytes = none ? 0 : M * K;
    if (scale_bytes) *scale_bytes = none ? 0 : M * (K / 128) * static_cast<int64_t>(sizeof(float));
    return DSNQ_OK;
}

extern "C" dsnq_status dsnq_block_scaled_fp8_gemm_dual_bf16a(
    int64_t M, int64_t K, const void* a_bf16, int64_t lda, int64_t N1, const void* w1_fp8, int64_t ldw1,
    const float* w1_scale, int64_t ld_w1scale, void* out1_bf16, int64_t ldo1, int64_t N2, const void* w2_fp8,
    int64_t ldw2, const float* w2_scale, int64_t ld_w2scale, void* out2_bf16, int64_t ldo2, void* a_fp8_ws,
    float* a_scale_ws, void* stream) {
    Consumer c0{N1, w1_fp8, ldw1, w1_scale, ld_w1scale, out1_bf16, ldo1};
    Consumer c1{N2, w2_fp8, ldw2, w2_scale, ld_w2scale, out2_bf16, ldo2};
    if (M < 0 || K <= 0 || N1 < 0 || N2 < 0) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > 4096) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    if (!a_bf16) return DSNQ_ERR_INVALID_ARG;
    dsnq_status st = check_consumer(c0, K);
    if (st != DSNQ_OK) return st;
    st = check_consumer(c1, K);
    if (st != DSNQ_OK) return st;
    if (N1 == 0 && N2 == 0) return DSNQ_OK;
    if (bf16a_in_gemm(M, K))   // a few decode rows: one launch, the kernel quantizes them itself
        return run_gemm(M, K, nullptr, 0, nullptr, DSNQ_SCALE_ROW_MAJOR, 0, c0, c1, stream, a_bf16, lda);
    // Otherwise quantize once into the caller's workspace, then the GEMM on
    // the pre-quantized pair (inside the GEMM every CTA would redo it).
    if (!a_fp8_ws || !a_scale_ws) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(a_fp8_ws, 16) || !aligned(a_scale_ws, 4)) return DSNQ_ERR_MISALIGNED;
    st = dsnq_group_quant_bf16(M, K, a_bf16, lda, 128, a_fp8_ws, K, a_scale_ws, DSNQ_SCALE_COL_MAJOR, M, stream);
    if (st != DSNQ_OK) return st;
    return run_gemm(M, K, a_fp8_ws, K, a_scale_ws, DSNQ_SCALE_COL_MAJOR, M, c0, c1, stream);
}

extern "C" dsnq_status dsnq_fused_norm_quant_gemm_dual(
    int64_t M, int64_t Kq, int64_t Kkv, const void* q, int64_t ldq, const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv, float eps, void* kv_out, int64_t ldkv_out, int64_t N1,
    const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale, void* out1_bf16, int64_t ldo1,
    int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale, int64_t ld_w2scale, void* out2_bf16,
    int64_t ldo2, void* q_fp8, float* q_scale, void* stream) {
    Consumer c0{N1, w1_fp8, ldw1, w1_scale, ld_w1scale, out1_bf16, ldo1};
    Consumer c1{N2, w2_fp8, ldw2, w2_scale, ld_w2scale, out2_bf16, ldo2};
    if (M < 0 || Kq <= 0 || Kkv <= 0 || N1 < 0 || N2 < 0) return DSNQ_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps > 3.4e38f) return DSNQ_ERR_INVALID_ARG;
    if (Kq % 128 != 0 || Kkv % 8 != 0 || Kq / 8 + Kkv / 8 > 512) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    if (!q || !kv || !gamma_q || !gamma_kv || !kv_out) return DSNQ_ERR_INVALID_ARG;
    if (ldq < Kq || ldkv < Kkv || ldkv_out < Kkv) return DSNQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(gamma_q, 16) || !aligned(gamma_kv, 16) ||
        !aligned(kv_out, 16) || ldq % 8 || ldkv % 8 || ldkv_out % 8)
        return DSNQ_ERR_MISALIGNED;
    if ((q_fp8 && !aligned(q_fp8, 16)) || (q_scale && !aligned(q_scale, 4))) return DSNQ_ERR_MISALIGNED;
    dsnq_status st = check_consumer(c0, Kq);
    if (st != DSNQ_OK) return st;
    st = check_consumer(c1, Kq);
    if (st != DSNQ_OK) return st;
    if (bf16a_in_gemm(M, Kq) && Kkv <= 2048) {
        // A few decode rows: one launch normalizes, quantizes and multiplies.
        const NormSide ns{gamma_q, kv, ldkv, gamma_kv, Kkv, eps, kv_out, ldkv_out, q_fp8, q_scale};
        if (N1 == 0 && N2 == 0) {
            // Nothing to multiply: the norm+quant alone (same outputs).
            if (!q_fp8 || !q_scale) return DSNQ_ERR_INVALID_ARG;
        } else {
            return run_gemm(M, Kq, nullptr, 0, nullptr, DSNQ_SCALE_ROW_MAJOR, 0, c0, c1, stream, q, ldq, &ns);
        }
    }
    // Otherwise the fused norm+quant kernel writes the pair, then the GEMM.
    if (!q_fp8 || !q_scale) return DSNQ_ERR_INVALID_ARG;
    st = dsnq_fused_dual_rmsnorm_group_quant(M, Kq, Kkv, q, ldq, kv, ldkv, gamma_q, gamma_kv, eps, 128, q_fp8, Kq,
                                             q_scale, DSNQ_SCALE_COL_MAJOR, M, kv_out, ldkv_out, stream);
    if (st != DSNQ_OK || (N1 == 0 && N2 == 0)) return st;
    return run_gemm(M, Kq, q_fp8, Kq, q_scale, DSNQ_SCALE_COL_MAJOR, M, c0, c1, stream);
}

extern "C" dsnq_status dsnq_debug_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0, w = 0, n = 0;
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
    // The index-check words of this unit and of the norm+quant unit.
    if (!take_debug_word(s, &w) || !take_norm_quant_debug_word(s, &n)) return DSNQ_ERR_CUDA;
    v |= w | n;
    if (v & kStatusTimeout) return DSNQ_ERR_TIMEOUT;
    return (v & kStatusBounds) ? DSNQ_ERR_BOUNDS : DSNQ_OK;
}
