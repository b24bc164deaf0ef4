// abi.cu -- the extern "C" entry points of moe_gb300.h: host-side argument
// checks, then asynchronous launches on the caller's stream.  Nothing here
// allocates, frees or synchronises.
#include <cuda_runtime.h>

#include "../../include/moe_gb300.h"
#include "launch.h"

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }
inline moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool sere_ok(const moe_sere_params* p, int N, int k) {
    return p->sim != nullptr && p->k_primary >= 1 && p->k_primary <= k && !(p->rho != p->rho) && N <= MOE_MAX_EXPERTS;
}

}  // namespace

extern "C" {

moe_status_t moe_route(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int R, int k,
                       uint32_t flags, float* logits, int32_t* ids, float* gates, const moe_sere_params* sere,
                       moe_dev_status* st, void* stream) {
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || R < 1 || R > MOE_MAX_RANKS || R > N || k < 1 || k > R)
        return MOE_ERR_INVALID_ARG;
    if (flags & ~(MOE_ROUTE_FROM_LOGITS | MOE_ROUTE_RENORM_TOPK)) return MOE_ERR_INVALID_ARG;
    if (sere != nullptr && (R != k || !sere_ok(sere, N, k))) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;  // nothing to rank; per-token pointers may be NULL
    if (logits == nullptr || ids == nullptr || gates == nullptr) return MOE_ERR_INVALID_ARG;
    const bool from_logits = (flags & MOE_ROUTE_FROM_LOGITS) != 0;
    if (!from_logits) {
        if (x == nullptr || w_router == nullptr || H < 1) return MOE_ERR_INVALID_ARG;
        if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
        if (x_dtype == MOE_DTYPE_BF16 && (H % 8 != 0)) return MOE_ERR_UNSUPPORTED;
        if (x_dtype == MOE_DTYPE_F32 && (H % 4 != 0)) return MOE_ERR_UNSUPPORTED;
        if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    }
    if (sere != nullptr) {
        if (R != k || !sere_ok(sere, N, k)) return MOE_ERR_INVALID_ARG;
        if (T > moe::kSereMaxT) return MOE_ERR_UNSUPPORTED;
    }
    cudaStream_t s = as_stream(stream);
    if (!from_logits) {
        cudaError_t e = moe::launch_router(x, x_dtype, w_router, T, H, N, logits, st, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    const bool renorm = (flags & MOE_ROUTE_RENORM_TOPK) != 0;
    if (sere != nullptr) return from_cuda(moe::launch_rank_sere(logits, T, N, k, renorm, ids, gates, *sere, st, s));
    return from_cuda(moe::launch_rank(logits, T, N, R, k, renorm, ids, gates, st, s));
}

moe_status_t moe_route_dispatch(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int k,
                                uint32_t flags, float* logits, int32_t* ids, float* gates,
                                const moe_sere_params* sere, int32_t* counts, int32_t* offsets, int32_t* row_token,
                                float* row_gate, int32_t* active, void* workspace, size_t ws_bytes,
                                moe_dev_status* st, void* stream) {
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_ROUTE_RENORM_TOPK) return MOE_ERR_INVALID_ARG;
    if (sere != nullptr && !sere_ok(sere, N, k)) return MOE_ERR_INVALID_ARG;
    if (counts == nullptr || offsets == nullptr || active == nullptr) return MOE_ERR_INVALID_ARG;
    if (T > moe::kRouteDispatchMaxT || T * k > moe::kRouteDispatchMaxSlots) return MOE_ERR_UNSUPPORTED;
    if (T == 0) {
        // no rows; with SERE the union bitmap and the statistics describe the
        // empty batch too (all zero), not the previous call's
        cudaStream_t s = as_stream(stream);
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * N, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (N + 1), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(active, 0, sizeof(int32_t) * (N + 1), s);
        if (e == cudaSuccess && sere != nullptr && sere->union_bitmap != nullptr)
            e = cudaMemsetAsync(sere->union_bitmap, 0, sizeof(uint32_t) * ((N + 31) / 32), s);
        if (e == cudaSuccess && sere != nullptr && sere->stats != nullptr)
            e = cudaMemsetAsync(sere->stats, 0, sizeof(int32_t) * 8, s);
        return from_cuda(e);
    }
    if (x == nullptr || w_router == nullptr || H < 1 || logits == nullptr || ids == nullptr || gates == nullptr ||
        row_token == nullptr || row_gate == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    if (x_dtype == MOE_DTYPE_BF16 && (H % 8 != 0)) return MOE_ERR_UNSUPPORTED;
    if (x_dtype == MOE_DTYPE_F32 && (H % 4 != 0)) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (workspace == nullptr || ws_bytes < static_cast<size_t>(moe::kRouteDispatchWs)) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_route_dispatch(x, x_dtype, w_router, T, H, N, k,
                                                (flags & MOE_ROUTE_RENORM_TOPK) != 0, logits, ids, gates, sere,
                                                counts, offsets, row_token, row_gate, active, workspace, false, st,
                                                as_stream(stream)));
}

moe_status_t moe_decode_layer(const void* x, const float* w_router, const void* w_gate, const void* w_up,
                              const void* w_down, int T, int H, int I, int N, int k, uint32_t route_flags,
                              uint32_t ffn_flags, const moe_sere_params* sere, float* logits, int32_t* ids,
                              float* gates, int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_gate,
                              int32_t* active, float* y, void* route_ws, size_t route_ws_bytes, void* ffn_ws,
                              size_t ffn_ws_bytes, moe_dev_status* st, void* stream) {
    if (N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N || H < 1 || I < 1)
        return MOE_ERR_INVALID_ARG;
    if ((route_flags & ~MOE_ROUTE_RENORM_TOPK) || (ffn_flags & ~MOE_FFN_ZERO_Y)) return MOE_ERR_INVALID_ARG;
    if (sere != nullptr && !sere_ok(sere, N, k)) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > moe::kDecodeMaxT || T * k > moe::kRouteDispatchMaxSlots) return MOE_ERR_UNSUPPORTED;
    if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (x == nullptr || w_router == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr ||
        logits == nullptr || ids == nullptr || gates == nullptr || counts == nullptr || offsets == nullptr ||
        row_token == nullptr || row_gate == nullptr || active == nullptr || y == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(N) * I > 0x7fffffffLL || static_cast<long long>(N) * H > 0x7fffffffLL)
        return MOE_ERR_UNSUPPORTED;
    if (route_ws == nullptr || route_ws_bytes < static_cast<size_t>(moe::kRouteDispatchWs)) return MOE_ERR_WORKSPACE;
    const size_t need = moe::ffn_workspace(T, H, I, N, k, MOE_DTYPE_BF16);
    if (ffn_ws == nullptr || ffn_ws_bytes < need) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(route_ws) & 255u) != 0 || (reinterpret_cast<uintptr_t>(ffn_ws) & 255u) != 0)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    cudaError_t e = moe::launch_route_dispatch(x, MOE_DTYPE_BF16, w_router, T, H, N, k,
                                               (route_flags & MOE_ROUTE_RENORM_TOPK) != 0, logits, ids, gates, sere,
                                               counts, offsets, row_token, row_gate, active, route_ws, true, st, s,
                                               moe::ffn_decode_one_wave_experts(T, I, N, k));
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const uint32_t* early = static_cast<const uint32_t*>(route_ws) + moe::kRouteDispatchEarlyWord;
    return from_cuda(moe::launch_ffn_decode(x, w_gate, w_up, w_down, T, H, I, N, k, offsets, row_token, row_gate,
                                            active, early, MOE_FFN_FUSE_COMBINE | ffn_flags, y, ffn_ws, st, s));
}

moe_status_t moe_reroute_sere(int32_t* ids, float* gates, int ld, int T, int N, int k, const moe_sere_params* sere,
                              moe_dev_status* st, void* stream) {
    if (ids == nullptr || gates == nullptr || sere == nullptr) return MOE_ERR_INVALID_ARG;
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N || ld < k)
        return MOE_ERR_INVALID_ARG;
    if (!sere_ok(sere, N, k)) return MOE_ERR_INVALID_ARG;
    if (T > moe::kSereMaxT) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    return from_cuda(moe::launch_sere(ids, gates, ld, T, N, k, *sere, st, as_stream(stream)));
}

size_t moe_workspace_size(int op, int T, int H, int I, int N, int k, int R, int capped, int dtype) {
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS) return 0;
    if (op == MOE_OP_DISPATCH) return moe::dispatch_workspace(T, N, k, R, capped != 0);
    if (op == MOE_OP_FFN) {
        if (H < 1 || I < 1) return 0;
        return moe::ffn_workspace(T, H, I, N, k, dtype);
    }
    if (op == MOE_OP_TOKEN_WEIGHTS) return moe::token_weights_workspace(T);
    if (op == MOE_OP_ROUTE_DISPATCH) return static_cast<size_t>(moe::kRouteDispatchWs);
    if (op == MOE_OP_CALIBRATE) {
        if (H < 1 || I < 1) return 0;
        return moe::calib_workspace(T, H, I, N);
    }
    return 0;
}

moe_status_t moe_dispatch_capacity(const int32_t* ids, const float* gates, int ld, int T, int N, int k, int R,
                                   const float* token_w, float capacity_factor, const int8_t* modality_bias,
                                   const float* r_v, int32_t* counts, int32_t* offsets,
                                   int32_t* row_token, float* row_gate, int32_t* active, int32_t* out_ids,
                                   float* out_gates, int32_t* slot_row, uint8_t* slot_status, int64_t* load_q,
                                   int64_t* cap_q, void* workspace, size_t ws_bytes, moe_dev_status* st,
                                   void* stream) {
    if (T < 0 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N) return MOE_ERR_INVALID_ARG;
    if (counts == nullptr || offsets == nullptr || active == nullptr ||
        ((ids == nullptr || gates == nullptr || row_token == nullptr || row_gate == nullptr) && T > 0))
        return MOE_ERR_INVALID_ARG;
    if (capacity_factor != capacity_factor) return MOE_ERR_INVALID_ARG;
    if (modality_bias != nullptr && (r_v == nullptr || !(capacity_factor > 0.f))) return MOE_ERR_INVALID_ARG;
    const bool capped = capacity_factor > 0.f;
    if (capped) {
        if (R < k || R > MOE_MAX_RANKS || R > N || ld < R) return MOE_ERR_INVALID_ARG;
        if (T > moe::kCapacityMaxT) return MOE_ERR_UNSUPPORTED;
    } else if (ld < k) {
        return MOE_ERR_INVALID_ARG;
    }
    const size_t need = moe::dispatch_workspace(T, N, k, R, capped);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return MOE_ERR_WORKSPACE;
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch(ids, gates, ld, T, N, k, R, token_w, capacity_factor, modality_bias, r_v,
                                          counts, offsets, row_token, row_gate, active, out_ids, out_gates, slot_row,
                                          slot_status, load_q, cap_q, workspace, st, as_stream(stream)));
}

moe_status_t moe_ffn_grouped(const void* x, int dtype, const void* w_gate, const void* w_up, const void* w_down,
                             int T, int H, int I, int N, int k, const int32_t* offsets, const int32_t* row_token,
                             const float* row_gate, const int32_t* active, uint32_t flags, float* out,
                             void* workspace, size_t ws_bytes, moe_dev_status* st, void* stream) {
    if (T < 0 || H < 1 || I < 1 || N < 1 || N > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_RANKS || k > N)
        return MOE_ERR_INVALID_ARG;
    if (flags & ~(MOE_FFN_FUSE_COMBINE | MOE_FFN_ZERO_Y)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_DTYPE_F32 && dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;  // no rows, nothing to write
    if (x == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr || offsets == nullptr ||
        row_token == nullptr || row_gate == nullptr || active == nullptr || out == nullptr)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (dtype == MOE_DTYPE_F32) {
        if (static_cast<long long>(H + I) * 4 > moe::kFfnF32MaxSmem) return MOE_ERR_UNSUPPORTED;
        return from_cuda(moe::launch_ffn_f32(static_cast<const float*>(x), static_cast<const float*>(w_gate),
                                             static_cast<const float*>(w_up), static_cast<const float*>(w_down), T,
                                             H, I, N, k, offsets, row_token, row_gate, active, flags, out, st, s));
    }
    if (dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    // tensor-map extents are 32-bit row counts
    if (static_cast<long long>(N) * I > 0x7fffffffLL || static_cast<long long>(N) * H > 0x7fffffffLL ||
        static_cast<long long>(T) * k > 0x7fffffffLL)
        return MOE_ERR_UNSUPPORTED;
    const size_t need = moe::ffn_workspace(T, H, I, N, k, dtype);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return MOE_ERR_WORKSPACE;
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_ffn_bf16(x, w_gate, w_up, w_down, T, H, I, N, k, offsets, row_token, row_gate,
                                          active, flags, out, workspace, st, s));
}

moe_status_t moe_similarity_calibrate(const void* x, int n, const void* w_gate, const void* w_up, const void* w_down,
                                      int H, int I, int N, float* sim, void* workspace, size_t ws_bytes,
                                      moe_dev_status* st, void* stream) {
    if (n < 1 || H < 1 || I < 1 || N < 2) return MOE_ERR_INVALID_ARG;
    if (x == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr || sim == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(sim))
        return MOE_ERR_INVALID_ARG;
    if (N > 128 || H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (static_cast<long long>(n) * N > 0x7fffffffLL || static_cast<long long>(n) * H > 0x7fffffffLL)
        return MOE_ERR_UNSUPPORTED;
    const size_t need = moe::calib_workspace(n, H, I, N);
    if (workspace == nullptr || ws_bytes < need) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_similarity(x, n, w_gate, w_up, w_down, H, I, N, sim, workspace, st,
                                            as_stream(stream)));
}

moe_status_t moe_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                               float eps, float* entropy, float* token_w, float* r_v, void* workspace,
                               size_t ws_bytes, moe_dev_status* st, void* stream) {
    if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !(delta == delta) || delta - delta != 0.f) return MOE_ERR_INVALID_ARG;   // eps > 0, delta finite
    if (T > (1 << 24)) return MOE_ERR_UNSUPPORTED;   // the fixed-point sums are sized for 2^24 tokens
    if (T == 0) {
        if (r_v == nullptr) return MOE_OK;
        return from_cuda(cudaMemsetAsync(r_v, 0, sizeof(float), as_stream(stream)));
    }
    if (x == nullptr || is_visual == nullptr || entropy == nullptr || token_w == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x)) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || ws_bytes < moe::token_weights_workspace(T)) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_token_weights(x, x_dtype, T, H, is_visual, delta, eps, entropy, token_w, r_v,
                                               workspace, st, as_stream(stream)));
}

moe_status_t moe_combine(const float* rows_out, const int32_t* slot_row, const float* slot_gate, int T, int H, int k,
                         float* y, void* stream) {
    if (T < 0 || H < 1 || k < 1 || k > MOE_MAX_RANKS) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (rows_out == nullptr || slot_row == nullptr || slot_gate == nullptr || y == nullptr)
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine(rows_out, slot_row, slot_gate, T, H, k, y, as_stream(stream)));
}

moe_status_t moe_residual_to_bf16(const float* x, void* y, long long n, void* stream) {
    if (n < 0 || n % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (x == nullptr || y == nullptr || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_residual_to_bf16(x, y, n, as_stream(stream)));
}

const char* moe_status_string(int code, int device) {
    if (device) {
        switch (code) {
            case MOE_DEV_OK: return "ok";
            case MOE_DEV_NONFINITE: return "non-finite router logit or token weight";
            case MOE_DEV_TIMEOUT: return "on-chip wait timed out";
            case MOE_DEV_BAD_INDEX: return "expert id or row index out of range";
            default: return "unknown device status";
        }
    }
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
        case MOE_ERR_CUDA: return "CUDA launch failed";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

}  // extern "C"
