// launch.h -- internal host-side launchers shared by the C-ABI layer (abi.cu)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

// Launches `kernel` on `s` with programmatic stream serialization, so that it
// may begin while its predecessor finishes; the kernel itself waits
// (griddepcontrol.wait) before touching memory the predecessor writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- routing (router.cu) ----
cudaError_t launch_router(const void* x, int x_dtype, const float* w_router, int T, int H, int N, float* logits,
                          moe_dev_status* st, cudaStream_t s);
cudaError_t launch_rank(const float* logits, int T, int N, int R, int k, bool renorm, int32_t* ids, float* gates,
                        moe_dev_status* st, cudaStream_t s);
cudaError_t launch_rank_sere(const float* logits, int T, int N, int k, bool renorm, int32_t* ids, float* gates,
                             const moe_sere_params& p, moe_dev_status* st, cudaStream_t s);
cudaError_t launch_sere(int32_t* ids, float* gates, int ld, int T, int N, int k, const moe_sere_params& p,
                        moe_dev_status* st, cudaStream_t s);
constexpr int kSereMaxT = 4096;

// ---- decode routing + dispatch in one launch (route_dispatch.cu) ----
constexpr int kRouteDispatchMaxT = 256;
constexpr int kRouteDispatchMaxSlots = 2048;   // T * k
constexpr int kRouteDispatchWs = 512;
// workspace word where the routing launch publishes its early experts for
// the decode FFN: a flag, then the bitmap (SERE's primary union P, else the
// union of all ranked experts), written as soon as ranking ends
constexpr int kRouteDispatchEarlyWord = 96;
// spec_union_max > 0 (with SERE and publish_early): when the batch's ranked
// union has at most that many experts, or at most twice that many while P
// has at most a third that many and the rest more than that many, the set
// published is the whole union instead of P, so the decode FFN streams every candidate's phase 1 at once
// (its SMs would otherwise idle); experts that then move lose only their
// phase 1
cudaError_t launch_route_dispatch(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int k,
                                  bool renorm, float* logits, int32_t* ids, float* gates, const moe_sere_params* sere,
                                  int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_gate,
                                  int32_t* active, void* ws, bool publish_early, moe_dev_status* st, cudaStream_t s,
                                  int spec_union_max = 0);

// ---- dispatch (dispatch.cu) ----
size_t dispatch_workspace(int T, int N, int k, int R, bool capped);
cudaError_t launch_dispatch(const int32_t* ids, const float* gates, int ld, int T, int N, int k, int R,
                            const float* token_w, float capacity_factor, const int8_t* modality_bias,
                            const float* r_v, int32_t* counts, int32_t* offsets, int32_t* row_token,
                            float* row_gate, int32_t* active, int32_t* out_ids, float* out_gates,
                            int32_t* slot_row, uint8_t* slot_status, int64_t* load_q, int64_t* cap_q, void* ws,
                            moe_dev_status* st, cudaStream_t s);
constexpr int kCapacityMaxT = 16384;

// ---- decode FFN, batches of up to 64 tokens (ffn_decode.cu) ----
constexpr int kDecodeMaxT = 64;
// batches the decode kernel runs (it stages every dispatch row, k <= 16)
inline bool ffn_use_decode(int T, int k) { return T >= 1 && T <= kDecodeMaxT && k <= MOE_MAX_RANKS; }
// token columns of the decode kernel's MMA operand for a batch of T tokens
inline int ffn_decode_nt(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : 64); }
// its counters (work counter, one per expert, three more) sit in a fixed
// region at the start of the workspace; the activations follow
inline size_t ffn_decode_ctr_bytes() { return 2304; }
long long ffn_decode_act_rows(int T, int N);
// phase-1 units per expert the decode kernel runs for this shape: I/64 half
// slices (64 gate and 64 up rows each)
int ffn_decode_units_per_expert(int T, int I, int N, int k);
// the most experts whose phase-1 units all fit one wave of the SMs
int ffn_decode_one_wave_experts(int T, int I, int N, int k);
// early: the routing launch's published early experts ([0] flag, then a
// bitmap), or nullptr to wait for the preceding launch at the start
cudaError_t launch_ffn_decode(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                              int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                              const int32_t* active, const uint32_t* early, uint32_t flags, float* out, void* ws,
                              moe_dev_status* st, cudaStream_t s);

// ---- FFN (ffn.cu) ----
// the fp32 kernel holds a row's x and activations in shared memory: (H + I) floats
constexpr int kFfnF32MaxSmem = 227 * 1024;
size_t ffn_workspace(int T, int H, int I, int N, int k, int dtype);
size_t ffn_workspace_zero_bytes(int T, int H, int N, int k, int dtype);
cudaError_t launch_ffn_f32(const float* x, const float* wg, const float* wu, const float* wd, int T, int H, int I,
                           int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                           const int32_t* active, uint32_t flags, float* out, moe_dev_status* st,
                           cudaStream_t s);
cudaError_t launch_ffn_bf16(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                            int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                            const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                            cudaStream_t s);
// ---- expert similarity from calibration tokens (calib.cu) ----
size_t calib_workspace(int n, int H, int I, int N);
cudaError_t launch_similarity(const void* x, int n, const void* wg, const void* wu, const void* wd, int H, int I,
                              int N, float* sim, void* ws, moe_dev_status* st, cudaStream_t s);

// ---- entropy-weighted token load (macs.cu) ----
size_t token_weights_workspace(int T);
cudaError_t launch_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                                 float eps, float* entropy, float* token_w, float* r_v, void* ws, moe_dev_status* st,
                                 cudaStream_t s);
cudaError_t launch_residual_to_bf16(const float* x, void* y, long long n, cudaStream_t s);

cudaError_t launch_combine(const float* rows_out, const int32_t* slot_row, const float* slot_gate, int T, int H,
                           int k, float* y, cudaStream_t s);

}  // namespace moe
