// Internal helpers shared by the CUDA translation units of libdsnq.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "dsnq.h"

namespace dsnq {

// Bits of the device status words read by dsnq_debug_status.
constexpr uint32_t kStatusTimeout = 1u;   // a bounded wait gave up
constexpr uint32_t kStatusBounds = 2u;    // a debug-build index check failed

// Test-hook flags (dsnq_debug_set).
constexpr uint32_t kInjectSkipLoad = 1u;          // the GEMM producer skips its first load
constexpr uint32_t kInjectBoundsSelfTest = 2u;    // debug build: one deliberate failed index check

// Test hooks and the wait bound, set by dsnq_debug_set (dsnq_api.cu).
uint32_t debug_inject_flags();
uint64_t debug_wait_timeout_ns();

// The status word of the norm+quant unit, read and cleared (norm_quant.cu).
bool take_norm_quant_debug_word(cudaStream_t s, unsigned int* v);

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Maps the launch outcome to a status; cudaGetLastError also clears the
// runtime's last-error slot so one failed call does not poison the next.
inline dsnq_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSNQ_OK : DSNQ_ERR_CUDA;
}

// Status of a launch made with cudaLaunchKernelEx (its own return value and
// the runtime's last-error slot, which is cleared).
inline dsnq_status launch_result(cudaError_t e) {
    const cudaError_t last = cudaGetLastError();
    return (e == cudaSuccess && last == cudaSuccess) ? DSNQ_OK : DSNQ_ERR_CUDA;
}

inline int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Programmatic dependent launch.  When enabled (the default; see
// dsnq_set_launch_overlap) every kernel is launched with programmatic stream
// serialization: it may be scheduled while the previous kernel of the stream
// still runs, sets up what depends on no input (barriers, tensor memory,
// descriptor prefetch), then waits in hardware (griddepcontrol.wait) until
// the previous kernel has completed and its writes are visible, before any
// thread reads global memory.
bool launch_overlap_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_overlap_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Wait until the kernels this grid depends on have completed and their
// memory operations are visible (returns at once for a plain launch).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel of the stream to be scheduled; it still waits for
// this grid's completion before reading anything.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Validated scale-buffer geometry: returns the effective ld or -1.
inline int64_t scale_ld(dsnq_scale_layout layout, int64_t M, int64_t G, int64_t ld) {
    if (layout == DSNQ_SCALE_ROW_MAJOR) return ld <= 0 ? G : (ld >= G ? ld : -1);
    if (layout == DSNQ_SCALE_COL_MAJOR) return ld <= 0 ? M : (ld >= M ? ld : -1);
    return -1;
}

}  // namespace dsnq
