// Device-side index checks of the debug build (compiled with -DDSNQ_DEBUG).
//
// Each translation unit that includes this header gets its own status word
// (the library is built without relocatable device code); dsnq_debug_status
// reads and clears every unit's word.  A failed check sets kStatusBounds in
// the word and makes the guarded access be skipped, so a wrong index is
// reported instead of touching memory outside the buffer; nothing traps.  In
// the release build every check is `true` and compiles away.
#pragma once

#include <cuda_runtime.h>

#include "dsnq_internal.h"

namespace dsnq {

static __device__ unsigned int g_debug_word;   // this translation unit's status word

__device__ __forceinline__ bool bounds_ok(bool ok) {
#ifdef DSNQ_DEBUG
    if (!ok) atomicOr(&g_debug_word, kStatusBounds);
    return ok;
#else
    (void)ok;
    return true;
#endif
}

// Test hook of the debug build (inject flag bit 1): one deliberate failed
// check per launch, with no memory access attached to it, so that the
// reporting path can be tested without a wrong index anywhere.
__device__ __forceinline__ void bounds_self_test(uint32_t inject) {
#ifdef DSNQ_DEBUG
    if ((inject & kInjectBoundsSelfTest) && blockIdx.x == 0 && threadIdx.x == 0) bounds_ok(false);
#else
    (void)inject;
#endif
}

// Reads and clears this unit's word (host; synchronizes `s`).
static inline bool take_debug_word(cudaStream_t s, unsigned int* v) {
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbolAsync(v, g_debug_word, sizeof(*v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_debug_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

}  // namespace dsnq
