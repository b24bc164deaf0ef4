// dispatch_static.cu -- moe_dispatch_capacity_static: the dispatch of
// moe_dispatch_capacity with its scratch memory in a fixed, file-scope device
// array instead of a caller-provided workspace, for callers that must not
// allocate device memory.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe_gb300.h"
#include "launch.h"

namespace {

// One array per device that loads this library, alive until the process exits.
static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_STATIC_DISPATCH_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The array's name in host code is only a host-side handle; its device
// address is looked up once per device, with that device current.
moe_status_t scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_dispatch_capacity_static(const int32_t* ids, const float* gates, int ld, int T, int N,
                                                     int k, int R, const float* token_w, float capacity_factor,
                                                     const int8_t* modality_bias, const float* r_v,
                                                     int32_t* counts, int32_t* offsets, int32_t* row_token,
                                                     float* row_gate, int32_t* active, int32_t* out_ids,
                                                     float* out_gates, int32_t* slot_row, uint8_t* slot_status,
                                                     int64_t* load_q, int64_t* cap_q, moe_dev_status* st,
                                                     void* stream) {
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N) return MOE_ERR_INVALID_ARG;
    if (T > MOE_STATIC_DISPATCH_MAX_T) return MOE_ERR_UNSUPPORTED;
    const bool capped = capacity_factor > 0.f;
    const size_t need = moe::dispatch_workspace(T, N, k, R, capped);
    if (need > sizeof(g_dispatch_scratch)) return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const moe_status_t s = scratch_for_current_device(&scratch);
    if (s != MOE_OK) return s;
    // The rest of the checks, and the kernels, are those of moe_dispatch_capacity;
    // it clears the parts of the scratch that must start at zero on every call.
    return moe_dispatch_capacity(ids, gates, ld, T, N, k, R, token_w, capacity_factor, modality_bias, r_v, counts,
                                 offsets, row_token, row_gate, active, out_ids, out_gates, slot_row, slot_status,
                                 load_q, cap_q, scratch, sizeof(g_dispatch_scratch), st, stream);
}
