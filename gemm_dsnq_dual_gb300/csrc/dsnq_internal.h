// Internal helpers shared by the CUDA translation units of libdsnq.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "dsnq.h"

namespace dsnq {

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Maps the launch outcome to a status; cudaGetLastError also clears the
// runtime's last-error slot so one failed call does not poison the next.
inline dsnq_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSNQ_OK : DSNQ_ERR_CUDA;
}

inline int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Validated scale-buffer geometry: returns the effective ld or -1.
inline int64_t scale_ld(dsnq_scale_layout layout, int64_t M, int64_t G, int64_t ld) {
    if (layout == DSNQ_SCALE_ROW_MAJOR) return ld <= 0 ? G : (ld >= G ? ld : -1);
    if (layout == DSNQ_SCALE_COL_MAJOR) return ld <= 0 ? M : (ld >= M ? ld : -1);
    return -1;
}

}  // namespace dsnq
