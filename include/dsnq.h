/*
 * dsnq.h - C ABI of libdsnq: the decode-step MLA latent pre-projection on
 * NVIDIA GB300 (sm_103a).
 *
 * The path has two kernels:
 *   1. a fused dual RMSNorm of the q-lora latent and the kv latent with fp32
 *      accumulation that, in the same pass, quantizes the normalized q latent
 *      per 1x128 group to FP8 E4M3FN with fp32 scales (single rounding) and
 *      writes the normalized kv latent as bf16
 *      (vLLM PR #53540, "Purpose": fused_qk_rmsnorm_group_quant replaces the
 *      Triton fused_q_kv_rmsnorm plus two per-1x128 quants);
 *   2. a W8A8 block-scaled FP8 GEMM that consumes the pre-quantized
 *      (q_fp8, q_scale) pair for one or two consumers, the attention wq_b and
 *      the indexer wq_b, with no second activation quantization
 *      (PR #53540 prhub summary, rocm.py snippet
 *      apply_pre_quantized_block_scaled_mm(A=x_fp8, B=weight, As=x_scale,
 *      Bs=weight_scale)).
 *
 * Conventions shared by every entry point:
 *   - Pointers named as device data are device pointers; the caller owns and
 *     allocates every buffer.  No entry point allocates, frees or
 *     synchronizes, except dsnq_debug_status, which synchronizes `stream`.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it.
 *   - Strides ("ld...") are in elements of the buffer's type, row-major.
 *   - bf16 is IEEE bfloat16 (uint16 storage), fp8 is OCP E4M3FN (uint8
 *     storage, bias 7, max 448, no infinities), fp32 is IEEE binary32.
 *   - Arguments are validated before anything is enqueued.  On any error the
 *     call enqueues nothing and returns the status; DSNQ_ERR_CUDA means a
 *     launch was attempted and the CUDA runtime reported an error (the
 *     runtime's last-error state is cleared).
 *   - M == 0 (N == 0 for the weight quantizer) is valid and enqueues
 *     nothing; the data pointers of such empty calls may be NULL.
 */
#ifndef DSNQ_H_
#define DSNQ_H_

#include <stdint.h>

#if defined(__GNUC__)
#define DSNQ_API __attribute__((visibility("default")))
#else
#define DSNQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSNQ_OK = 0,
    DSNQ_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld too small, bad enum */
    DSNQ_ERR_MISALIGNED = 2,    /* base or stride not aligned as the call requires */
    DSNQ_ERR_UNSUPPORTED = 3,   /* a valid request outside the shapes implemented */
    DSNQ_ERR_CUDA = 4,          /* the CUDA runtime reported an error */
    DSNQ_ERR_TIMEOUT = 5,       /* a bounded device wait gave up (see dsnq_debug_status) */
    DSNQ_ERR_BOUNDS = 6         /* debug build: a device index check failed (see dsnq_debug_status) */
} dsnq_status;

/* Scale layout of the per-1x128 activation scales, logical shape [M, G]
 * with G = K / 128 (sglang PR #27289, "transpose_scale": the column-major
 * form is the transposed copy viewed with strides (1, M)).
 *   DSNQ_SCALE_ROW_MAJOR: element (m, g) at m * ld_scale + g, ld_scale >= G.
 *   DSNQ_SCALE_COL_MAJOR: element (m, g) at g * ld_scale + m, ld_scale >= M. */
typedef enum {
    DSNQ_SCALE_ROW_MAJOR = 0,
    DSNQ_SCALE_COL_MAJOR = 1
} dsnq_scale_layout;

/* Human-readable name of a status.  Never NULL. */
DSNQ_API const char* dsnq_status_string(dsnq_status status);

/* Library version as major*10000 + minor*100 + patch. */
DSNQ_API int32_t dsnq_version(void);

/*
 * Shapes of the quantized outputs, mirroring the custom op's fake (meta)
 * implementation (PR #53540 prhub summary, _fused_mla_dual_rms_norm_group_quant_fake:
 * q_out [M, Nq] fp8, q_scale [M, Nq/group] fp32).
 *   n_scale_elems   <- number of fp32 slots the scale buffer needs at the
 *                      default ld (M*G for both layouts);
 *   default_ld_scale <- G (row-major) or M (column-major).
 * Either output pointer may be NULL.  Pure host function.
 * Errors: INVALID_ARG (M < 0, Kq <= 0, bad layout), UNSUPPORTED (group != 128
 * or Kq % 128 != 0).
 */
DSNQ_API dsnq_status dsnq_quant_output_sizes(int64_t M, int64_t Kq, int32_t group,
                                    dsnq_scale_layout layout,
                                    int64_t* n_scale_elems, int64_t* default_ld_scale);

/*
 * Fused dual RMSNorm + per-1x128 FP8 group quant
 * (PR #53540, "Purpose" and the prhub summary's _aiter_ops.py snippet,
 * op fused_mla_dual_rms_norm_group_quant(q, q_weight, kv, kv_weight,
 * q_epsilon, kv_epsilon, group_size, transpose_scale)).
 *
 * For each token row m:
 *   r_q  = 1 / sqrt(mean_k q[m,k]^2 + eps)    (fp32 accumulation, over Kq)
 *   r_kv = 1 / sqrt(mean_k kv[m,k]^2 + eps)   (over Kkv)
 *   xq   = q * r_q * gamma_q,  xkv = kv * r_kv * gamma_kv   (fp32)
 *   per group g of 128 columns of xq: amax = max |xq|,
 *     q_scale(m, g) = amax / 448  (fp32; 0 when amax == 0),
 *     q_fp8[m, k]   = e4m3_rn_satfinite(fp32(xq[m,k] / q_scale(m, g)))  (0 when amax == 0),
 *                     the quotient taken on the fp32 values (single rounding)
 *   kv_out[m, k]  = bf16_rn(xkv[m, k])
 * One eps serves both latents (the model passes the same self.eps to both).
 *
 * Arguments (device pointers unless stated):
 *   M, Kq, Kkv : rows, q width (multiple of 128), kv width (multiple of 8);
 *                Kq/8 + Kkv/8 <= 512.
 *   q, ldq     : bf16 [M, Kq] with row stride ldq >= Kq; may be a column
 *                slice of a wider buffer (the split view of the fused
 *                projection output: ldq = 2112).
 *   kv, ldkv   : bf16 [M, Kkv], row stride ldkv >= Kkv; may alias the same
 *                buffer as q (read only).
 *   gamma_q, gamma_kv : bf16 [Kq] and [Kkv].
 *   eps        : host fp32, finite and >= 0 (eps == 0 with an all-zero row
 *                yields NaN, as the formula does).
 *   group      : must be 128.
 *   q_fp8, ldq_out : e4m3 [M, Kq] output, row stride ldq_out >= Kq.
 *   q_scale, layout, ld_scale : fp32 scale output in the given layout;
 *                ld_scale <= 0 selects the default (G or M).
 *   kv_out, ldkv_out : bf16 [M, Kkv] output, row stride ldkv_out >= Kkv.
 * Alignment (DSNQ_ERR_MISALIGNED otherwise): q, kv, gamma_q, gamma_kv and
 * kv_out 16-byte aligned with ldq, ldkv, ldkv_out multiples of 8; q_fp8
 * 8-byte aligned with ldq_out a multiple of 8; q_scale 4-byte aligned.
 * Outputs must not overlap inputs or each other.
 */
DSNQ_API dsnq_status dsnq_fused_dual_rmsnorm_group_quant(
    int64_t M, int64_t Kq, int64_t Kkv,
    const void* q, int64_t ldq,
    const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv,
    float eps, int32_t group,
    void* q_fp8, int64_t ldq_out,
    float* q_scale, dsnq_scale_layout layout, int64_t ld_scale,
    void* kv_out, int64_t ldkv_out,
    void* stream);

/*
 * Single-latent RMSNorm + per-1x128 FP8 group quant: the fused call for one
 * latent, as in the DeepSeek MLA pattern that normalizes one latent before
 * its block-scaled FP8 projection (sglang PR #27289, fused_rms_fp8_group_quant
 * with transpose_scale).  Same formulas as the q part of the fused call:
 *   r = 1 / sqrt(mean_k x[m,k]^2 + eps),  xn = x * r * gamma  (fp32),
 *   x_scale(m, g) = amax_g / 448,  x_fp8 = e4m3_rn_satfinite(fp32(xn / x_scale)).
 * Arguments: M rows; K (multiple of 128, <= 4096); x bf16 [M, K] with row
 * stride ldx (multiple of 8, may be a column slice of a wider buffer);
 * gamma bf16 [K]; eps, group, x_fp8/ldx_out, x_scale/layout/ld_scale as in
 * the fused call.  Alignment and error rules as in the fused call.
 */
DSNQ_API dsnq_status dsnq_rmsnorm_group_quant(
    int64_t M, int64_t K,
    const void* x, int64_t ldx, const void* gamma,
    float eps, int32_t group,
    void* x_fp8, int64_t ldx_out,
    float* x_scale, dsnq_scale_layout layout, int64_t ld_scale,
    void* stream);

/*
 * Baseline step 1 of the unfused sequence the fusion replaces: the dual
 * RMSNorm alone, both latents written as bf16 (PR #53540 prhub summary,
 * shared-path snippet: fused_q_kv_rmsnorm(qr, kv, q_norm.weight,
 * kv_norm.weight, eps)).  Same formulas, arguments and alignment rules as
 * the fused call; q_out is bf16 [M, Kq] with row stride ldq_out (multiple of 8).
 */
DSNQ_API dsnq_status dsnq_dual_rmsnorm_bf16(
    int64_t M, int64_t Kq, int64_t Kkv,
    const void* q, int64_t ldq,
    const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv,
    float eps,
    void* q_out, int64_t ldq_out,
    void* kv_out, int64_t ldkv_out,
    void* stream);

/*
 * Baseline step 2: per-1x128 dynamic quant of a bf16 tensor to E4M3FN with
 * fp32 scales (PR #53540, "Purpose": the aiter per-1x128 quant of the bf16
 * q-lora; sglang PR #27289, aiter_per1x128_quant with transpose_scale).
 * x is bf16 [M, K] (row stride ldx, multiple of 8, 16-byte aligned base),
 * K a multiple of 128 and at most 4096.  Outputs as in the fused call.
 */
DSNQ_API dsnq_status dsnq_group_quant_bf16(
    int64_t M, int64_t K,
    const void* x, int64_t ldx, int32_t group,
    void* x_fp8, int64_t ldx_out,
    float* x_scale, dsnq_scale_layout layout, int64_t ld_scale,
    void* stream);

/*
 * Load-time weight preparation: per-128x128-block quantization of an fp32
 * weight [N, K] to E4M3FN codes with fp32 block scales
 * (sglang PR #27289, aiter_w8a8_block_fp8_linear: block_size [128, 128] and
 * one fp32 weight_scale per block).  Per block: s = amax / 448 (0 when
 * amax == 0), code = e4m3_rn_satfinite(w * 448 / amax).
 *   w, ldw       : fp32 [N, K], ldw >= K, 16-byte aligned, ldw % 4 == 0.
 *   w_fp8, ldw_out : e4m3 [N, K] output, ldw_out >= K, ldw_out % 16 == 0,
 *                    16-byte aligned.
 *   w_scale, ld_wscale : fp32 [ceil(N/128), K/128], ld_wscale >= K/128.
 * K must be a multiple of 128.
 */
DSNQ_API dsnq_status dsnq_quantize_weight_block128(
    int64_t N, int64_t K,
    const float* w, int64_t ldw,
    void* w_fp8, int64_t ldw_out,
    float* w_scale, int64_t ld_wscale,
    void* stream);

/*
 * W8A8 block-scaled FP8 GEMM on pre-quantized activations
 * (PR #53540 prhub summary, rocm.py snippet apply_pre_quantized_block_scaled_mm
 * -> kernel.apply_block_scaled_mm(A=x_fp8, B=weight, As=x_scale,
 * Bs=weight_scale), output cast to the model dtype; sglang PR #27289,
 * aiter_w8a8_block_fp8_linear, input_scale branch):
 *
 *   out[m, n] = bf16_rn( sum_{kb} sa(m, kb) * sw[n/128, kb]
 *                        * sum_{k in block kb} a[m, k] * w[n, k] )
 *
 * with fp32 accumulation of each 128-wide K block on the tensor cores and the
 * scaled sum over K blocks in fp32.
 *   a_fp8, lda : e4m3 [M, K], lda >= K, lda % 16 == 0, 16-byte aligned.
 *   a_scale, a_scale_layout, ld_ascale : fp32 activation scales, logical
 *                [M, K/128], in either layout (ld_ascale <= 0 = default).
 *   w_fp8, ldw : e4m3 [N, K] (K-major, one output feature per row),
 *                ldw >= K, ldw % 16 == 0, 16-byte aligned.
 *   w_scale, ld_wscale : fp32 [ceil(N/128), K/128], ld_wscale >= K/128.
 *   out_bf16, ldo : bf16 [M, N], ldo >= N, ldo % 8 == 0, 16-byte aligned.
 * K must be a multiple of 128 and at most 8192 (DSNQ_ERR_UNSUPPORTED otherwise,
 * before anything is enqueued) and N a multiple of 16; every M >= 1 and every
 * such K is served (dsnq_gemm_plan names the kernel variant a call takes).
 * The output must not overlap the inputs.
 */
DSNQ_API dsnq_status dsnq_block_scaled_fp8_gemm(
    int64_t M, int64_t N, int64_t K,
    const void* a_fp8, int64_t lda,
    const float* a_scale, dsnq_scale_layout a_scale_layout, int64_t ld_ascale,
    const void* w_fp8, int64_t ldw,
    const float* w_scale, int64_t ld_wscale,
    void* out_bf16, int64_t ldo,
    void* stream);

/*
 * Two consumers of one pre-quantized activation in a single launch: the
 * attention wq_b (N1) and the indexer wq_b (N2) both read the same
 * (a_fp8, a_scale) pair, so the activation is quantized once
 * (PR #53540, "Purpose": both wq_b GEMMs consume the pre-quantized pair and
 * skip their own input quant).  Each consumer obeys the rules of
 * dsnq_block_scaled_fp8_gemm; N2 == 0 reduces to the single call.
 */
DSNQ_API dsnq_status dsnq_block_scaled_fp8_gemm_dual(
    int64_t M, int64_t K,
    const void* a_fp8, int64_t lda,
    const float* a_scale, dsnq_scale_layout a_scale_layout, int64_t ld_ascale,
    int64_t N1, const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale,
    void* out1_bf16, int64_t ldo1,
    int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale, int64_t ld_w2scale,
    void* out2_bf16, int64_t ldo2,
    void* stream);

/*
 * Host-only query (no CUDA call): the kernel variant dsnq_block_scaled_fp8_gemm
 * and dsnq_block_scaled_fp8_gemm_dual launch for M activation rows and
 * reduction length K, and its dynamic shared memory per CTA in bytes.  No
 * counterpart in the published method: it describes this implementation.
 *   variant : 1 / 2 / 3  decode, M <= 16 / 32 / 64: swap-AB, the weights fill
 *                        the MMA's 128 rows and the tokens are its N;
 *             4          128 x 128 tiles, five-stage operand ring (64 < M < 256,
 *                        K <= 4096);
 *             5          128 x 128 tiles, three-stage ring (M > 64, K > 4096:
 *                        the ring gives way to the scale slots of long K);
 *             6          256 x 256 tiles on CTA pairs (M >= 256, K <= 4096).
 *   M == 0 reports variant 0 and 0 bytes (nothing would be launched).
 * DSNQ_ERR_UNSUPPORTED when no variant serves (M, K): K not a multiple of
 * 128 or K > 8192.  DSNQ_ERR_INVALID_ARG for M < 0 or K <= 0.  Either output
 * pointer may be NULL.
 */
DSNQ_API dsnq_status dsnq_gemm_plan(int64_t M, int64_t K, int32_t* variant, int64_t* smem_bytes);

/*
 * Host-only query: the workspace dsnq_block_scaled_fp8_gemm_dual_bf16a needs
 * for M rows of K bf16 activations, as the byte sizes of its two buffers
 * (codes, scales); both 0 when the call quantizes inside the GEMM and reads
 * no workspace.  No counterpart in the published method.
 * DSNQ_ERR_UNSUPPORTED for K not a multiple of 128 or K > 4096;
 * DSNQ_ERR_INVALID_ARG for M < 0 or K <= 0.  Either output may be NULL.
 */
DSNQ_API dsnq_status dsnq_bf16a_workspace_bytes(int64_t M, int64_t K, int64_t* code_bytes,
                                                int64_t* scale_bytes);

/*
 * The dual GEMM for callers without a pre-quantized pair: bf16 activations
 * are quantized per 1x128 group on the fly, then multiplied as in
 * dsnq_block_scaled_fp8_gemm_dual (sglang PR #27289, aiter_w8a8_block_fp8_linear:
 * when no input_scale is given, the input is quantized in the current step by
 * the per-1x128 quant kernel before the block-scaled GEMM).  The quantization
 * is that of dsnq_group_quant_bf16: per group of 128 values of a row,
 * sa = fp32(amax / 448) and code = e4m3_rn_satfinite(fp32(a / sa)).
 *   a_bf16, lda : bf16 [M, K], lda >= K, lda % 8 == 0, 16-byte aligned.
 *   consumers   : as in dsnq_block_scaled_fp8_gemm_dual (N2 == 0: one consumer).
 *   a_fp8_ws, a_scale_ws : caller-owned workspace for the quantized pair,
 *                 M*K bytes (16-byte aligned) and M*(K/128) floats (4-byte
 *                 aligned, written column-major).  Unused, and may be NULL,
 *                 when M <= 8, K <= 2048 and M * ceil(K/256) <= 40 (M <= 6
 *                 at K = 1536): there one launch quantizes the activations
 *                 inside the GEMM, into shared memory.  Every CTA quantizes
 *                 all M rows, so larger batches run the quant kernel into the
 *                 workspace and then the GEMM (two launches).
 * K must be a multiple of 128 and at most 4096.  DSNQ_ERR_INVALID_ARG when the
 * workspace is needed and NULL.  The outputs must not overlap the inputs or
 * the workspace.
 */
DSNQ_API dsnq_status dsnq_block_scaled_fp8_gemm_dual_bf16a(
    int64_t M, int64_t K,
    const void* a_bf16, int64_t lda,
    int64_t N1, const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale,
    void* out1_bf16, int64_t ldo1,
    int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale, int64_t ld_w2scale,
    void* out2_bf16, int64_t ldo2,
    void* a_fp8_ws, float* a_scale_ws,
    void* stream);

/*
 * dsnq_block_scaled_fp8_gemm_dual_bf16a without a workspace argument: the
 * quantized pair goes to a device array inside the library (2048 x 2048
 * codes and their scales), so the call allocates nothing.  No counterpart in
 * the published method: an interface variant of this implementation.
 * M <= 2048 and K <= 2048 with K a multiple of 128 (DSNQ_ERR_UNSUPPORTED
 * otherwise); other arguments and rules as in
 * dsnq_block_scaled_fp8_gemm_dual_bf16a.  Calls that use the array (those
 * outside the one-launch case) share it: on one device they must be ordered,
 * e.g. issued to one stream, since calls that overlap on the GPU race on it.
 * The first call on a device looks the array's address up (which may load
 * the library's device code), in relaxed capture mode for the calling thread,
 * so that first call may also be made while a stream is being captured.
 */
DSNQ_API dsnq_status dsnq_block_scaled_fp8_gemm_dual_bf16a_static(
    int64_t M, int64_t K,
    const void* a_bf16, int64_t lda,
    int64_t N1, const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale,
    void* out1_bf16, int64_t ldo1,
    int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale, int64_t ld_w2scale,
    void* out2_bf16, int64_t ldo2,
    void* stream);

/*
 * The whole pre-projection in one call: the fused dual RMSNorm + per-1x128
 * quant of dsnq_fused_dual_rmsnorm_group_quant, then the dual block-scaled
 * GEMM of dsnq_block_scaled_fp8_gemm_dual on the quantized q latent.  Same
 * formulas; kv_out as in the fused call.  No counterpart in the published
 * method, which launches the two steps separately: for a few decode rows
 * (M <= 8, Kq <= 2048, Kkv <= 2048 and M * ceil(Kq/256) <= 40, i.e. M <= 6
 * at Kq = 1536) one launch normalizes and quantizes the rows inside the GEMM,
 * where both steps are bound by latency; otherwise the fused norm+quant
 * kernel writes (q_fp8, q_scale) and the GEMM reads them.
 *   M, Kq, Kkv, q/ldq, kv/ldkv, gamma_q, gamma_kv, eps, kv_out/ldkv_out :
 *                 as in dsnq_fused_dual_rmsnorm_group_quant.
 *   consumers   : as in dsnq_block_scaled_fp8_gemm_dual (K = Kq).
 *   q_fp8, q_scale : the quantized pair, e4m3 [M, Kq] with row stride Kq
 *                 (16-byte aligned) and fp32 scales column-major with ld M
 *                 (4-byte aligned).  Required outside the one-launch case
 *                 (DSNQ_ERR_INVALID_ARG when NULL); there they are optional
 *                 outputs (NULL: not written).
 * Alignment and error rules as in the two calls it combines.
 */
DSNQ_API dsnq_status dsnq_fused_norm_quant_gemm_dual(
    int64_t M, int64_t Kq, int64_t Kkv,
    const void* q, int64_t ldq,
    const void* kv, int64_t ldkv,
    const void* gamma_q, const void* gamma_kv,
    float eps,
    void* kv_out, int64_t ldkv_out,
    int64_t N1, const void* w1_fp8, int64_t ldw1, const float* w1_scale, int64_t ld_w1scale,
    void* out1_bf16, int64_t ldo1,
    int64_t N2, const void* w2_fp8, int64_t ldw2, const float* w2_scale, int64_t ld_w2scale,
    void* out2_bf16, int64_t ldo2,
    void* q_fp8, float* q_scale,
    void* stream);

/*
 * Device status words.  Kernels with bounded waits (the GEMM's mbarrier
 * waits) record a timeout there instead of hanging.  In the debug build
 * (libdsnq_debug.so, compiled with DSNQ_DEBUG) every kernel also checks the
 * indices of its memory accesses against the buffer extents its arguments
 * describe; a failed check skips the access and records a bounds error.
 * This call synchronizes `stream`, reads the words of the current device,
 * clears them and returns DSNQ_OK, DSNQ_ERR_TIMEOUT, DSNQ_ERR_BOUNDS (a
 * timeout takes precedence when both are recorded), or DSNQ_ERR_CUDA if the
 * synchronize failed.  No counterpart in the published method.
 */
DSNQ_API dsnq_status dsnq_debug_status(void* stream);

/* 1 when this library is the debug build (device index checks), else 0. */
DSNQ_API int32_t dsnq_debug_build(void);

/*
 * Launch overlap (programmatic dependent launch), on by default; affects
 * later launches of every entry point on all devices of this process.
 * When on, each kernel is launched so that it may be scheduled while the
 * previous kernel of its stream is still running: it prepares what reads no
 * input (barriers, tensor memory, descriptors) and then waits in hardware
 * until that kernel has completed and its writes are visible, before reading
 * any argument buffer.  Results are identical either way; only the gap
 * between dependent launches (a decode step's norm+quant and GEMM, say)
 * shrinks.  enable = 0 restores plain stream ordering.  No counterpart in the
 * published method: a launch property of this implementation.
 */
DSNQ_API void dsnq_set_launch_overlap(int32_t enable);

/*
 * Test hooks (affect later launches on all devices of this process).
 * wait_timeout_ns bounds every device wait (0 restores the default of 2 s).
 * inject_flags bit 0 makes the GEMM's producer skip the first stage's load,
 * so the consumer's wait on it must run out: the kernel then records
 * DSNQ_ERR_TIMEOUT, releases its tensor memory and returns.  Bit 1 (debug
 * build only; ignored otherwise) makes every launch record one failed index
 * check that guards no access, to test the reporting path.
 */
DSNQ_API void dsnq_debug_set(uint32_t inject_flags, uint64_t wait_timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DSNQ_H_ */
