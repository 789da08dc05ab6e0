// dsnq_block_scaled_fp8_gemm_dual_bf16a_static: the bf16-activation dual GEMM
// with its quantized-pair workspace in a file-scope device array instead of
// a caller buffer, so that the call allocates nothing and takes no workspace
// argument.  The array is part of the library's device image; its address on
// each device is looked up once (cudaGetSymbolAddress) and cached.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dsnq_internal.h"

namespace dsnq {
namespace {

constexpr int64_t kScratchRows = 2048;
constexpr int64_t kScratchK = 2048;
static __device__ __align__(256) uint8_t g_scratch_codes[kScratchRows * kScratchK];
static __device__ __align__(256) float g_scratch_scales[kScratchRows * (kScratchK / 128)];

constexpr int kMaxDevices = 64;
struct ScratchPtrs {
    void* codes;
    float* scales;
};
std::mutex g_lock;
ScratchPtrs g_ptrs[kMaxDevices];
std::atomic<bool> g_ready[kMaxDevices];

// The arrays' addresses on the current device (looked up once per device).
bool scratch_ptrs(ScratchPtrs* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    if (!g_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_lock);
        if (!g_ready[dev].load(std::memory_order_relaxed)) {
            ScratchPtrs p{};
            // The lookup may load the library's device code; in relaxed
            // capture mode for this thread it is allowed while a stream of
            // the caller is being captured (the first call inside a graph).
            cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
            cudaThreadExchangeStreamCaptureMode(&mode);
            const bool found = cudaGetSymbolAddress(&p.codes, g_scratch_codes) == cudaSuccess &&
                               cudaGetSymbolAddress(reinterpret_cast<void**>(&p.scales), g_scratch_scales) == cudaSuccess;
            cudaThreadExchangeStreamCaptureMode(&mode);   // the caller's mode back
            if (!found) {
                cudaGetLastError();
                return false;
            }
            g_ptrs[dev] = p;
            g_ready[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_ptrs[dev];
    return true;
}

}  // namespace
}  // namespace dsnq

extern "C" dsnq_status dsnq_block_scaled_fp8_gemm_dual_bf16a_static(
    int64_t M, int64_t K, const void* a_bf16, int64_t lda, int64_t N1, const void* w1_fp8, int64_t ldw1,
    const float* w1_scale, int64_t ld_w1scale, void* out1_bf16, int64_t ldo1, int64_t N2, const void* w2_fp8,
    int64_t ldw2, const float* w2_scale, int64_t ld_w2scale, void* out2_bf16, int64_t ldo2, void* stream) {
    using namespace dsnq;
    // The same size checks as the workspace entry, before the early returns,
    // so both report the same status for the same bad input.
    if (M < 0 || K <= 0 || N1 < 0 || N2 < 0) return DSNQ_ERR_INVALID_ARG;
    if (K % 128 != 0) return DSNQ_ERR_UNSUPPORTED;
    if (M > kScratchRows || K > kScratchK) return DSNQ_ERR_UNSUPPORTED;
    if (M == 0) return DSNQ_OK;
    ScratchPtrs ws{};
    if (!scratch_ptrs(&ws)) return DSNQ_ERR_CUDA;
    return dsnq_block_scaled_fp8_gemm_dual_bf16a(M, K, a_bf16, lda, N1, w1_fp8, ldw1, w1_scale, ld_w1scale, out1_bf16,
                                                 ldo1, N2, w2_fp8, ldw2, w2_scale, ld_w2scale, out2_bf16, ldo2, ws.codes,
                                                 ws.scales, stream);
}
