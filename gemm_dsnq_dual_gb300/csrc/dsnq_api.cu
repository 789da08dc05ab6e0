// Host-only entry points of libdsnq: status strings, version and the shape
// helper mirroring the fused op's fake (meta) implementation
// (vLLM PR #53540 prhub summary, _fused_mla_dual_rms_norm_group_quant_fake:
// q_out [M, Nq] fp8 and q_scale [M, Nq / group_size] fp32).

#include <atomic>

#include "dsnq_internal.h"

extern "C" const char* dsnq_status_string(dsnq_status status) {
    switch (status) {
        case DSNQ_OK: return "DSNQ_OK";
        case DSNQ_ERR_INVALID_ARG: return "DSNQ_ERR_INVALID_ARG";
        case DSNQ_ERR_MISALIGNED: return "DSNQ_ERR_MISALIGNED";
        case DSNQ_ERR_UNSUPPORTED: return "DSNQ_ERR_UNSUPPORTED";
        case DSNQ_ERR_CUDA: return "DSNQ_ERR_CUDA";
        case DSNQ_ERR_TIMEOUT: return "DSNQ_ERR_TIMEOUT";
        case DSNQ_ERR_BOUNDS: return "DSNQ_ERR_BOUNDS";
    }
    return "DSNQ_ERR_UNKNOWN";
}

extern "C" int32_t dsnq_version(void) { return 100; }  // 0.1.0

namespace {
std::atomic<int> g_launch_overlap{1};
std::atomic<uint32_t> g_inject{0};
std::atomic<uint64_t> g_timeout_ns{0};
}

bool dsnq::launch_overlap_enabled() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }
uint32_t dsnq::debug_inject_flags() { return g_inject.load(std::memory_order_relaxed); }
uint64_t dsnq::debug_wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

extern "C" void dsnq_debug_set(uint32_t inject_flags, uint64_t wait_timeout_ns) {
    g_inject.store(inject_flags);
    g_timeout_ns.store(wait_timeout_ns);
}

extern "C" int32_t dsnq_debug_build(void) {
#ifdef DSNQ_DEBUG
    return 1;
#else
    return 0;
#endif
}

extern "C" void dsnq_set_launch_overlap(int32_t enable) {
    g_launch_overlap.store(enable ? 1 : 0, std::memory_order_relaxed);
}

extern "C" dsnq_status dsnq_quant_output_sizes(int64_t M, int64_t Kq, int32_t group, dsnq_scale_layout layout,
                                               int64_t* n_scale_elems, int64_t* default_ld_scale) {
    if (M < 0 || Kq <= 0) return DSNQ_ERR_INVALID_ARG;
    if (layout != DSNQ_SCALE_ROW_MAJOR && layout != DSNQ_SCALE_COL_MAJOR) return DSNQ_ERR_INVALID_ARG;
    if (group != 128 || Kq % 128 != 0) return DSNQ_ERR_UNSUPPORTED;
    const int64_t G = Kq / group;
    if (n_scale_elems) *n_scale_elems = M * G;
    if (default_ld_scale) *default_ld_scale = layout == DSNQ_SCALE_ROW_MAJOR ? G : M;
    return DSNQ_OK;
}
