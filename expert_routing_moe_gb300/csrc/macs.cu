// macs.cu -- entropy-weighted token load for the capacity dispatch.
//
// "MACS: Modality-Aware Capacity Scaling for Efficient Multimodal MoE
// Inference", sec. 3.2 Eqs. (4)-(5) and sec. 3.3 Eq. (7): each token's
// feature vector z (here the layer's input row, D = H) gives p = Softmax(z)
// and its Shannon entropy; over the batch's visual tokens the entropies are
// z-scored (population statistics) and mapped to a load weight
// w = sigmoid(-delta * Htilde); text tokens weigh 1.  The effective visual
// ratio R_v = sum_vis w / sum_all w.
//
// Kernel 1: one warp per token, H = ln Z - (sum e_d (z_d - m)) / Z with
// m = max z and e_d = exp(z_d - m), fixed lane order and xor butterfly.
// Kernel 2: one CTA; the statistics and R_v are summed in double in a fixed
// order (per-thread strided sums, then a fixed tree), so results are
// reproducible bit for bit; each token's sigmoid is evaluated in fp32 (one
// SM evaluating T double-precision exponentials would dominate the call).
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(u[j] << 16);
        v[2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename XT>
__global__ void __launch_bounds__(256) token_entropy_kernel(const XT* __restrict__ x, int T, int H,
                                                            float* __restrict__ entropy, moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const XT* row = x + static_cast<size_t>(t) * H;
    float m = -INFINITY;
    bool finite = true;
    for (int h = lane * 8; h < H; h += 256) {
        float v[8];
        load8(row + h, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            finite &= isfinite(v[j]);
            m = fmaxf(m, v[j]);
        }
    }
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    float Z = 0.f, S1 = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
        float v[8];
        load8(row + h, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float d = v[j] - m;
            const float e = expf(d);
            Z += e;
            S1 = fmaf(e, d, S1);
        }
    }
    for (int off = 16; off >= 1; off >>= 1) {
        Z += __shfl_xor_sync(kFull, Z, off);
        S1 += __shfl_xor_sync(kFull, S1, off);
    }
    const bool all_finite = __all_sync(kFull, finite);
    if (lane == 0) {
        entropy[t] = logf(Z) - S1 / Z;
        if (!all_finite) report(st, MOE_DEV_NONFINITE, t);
    }
}

// Sum over the block in double, fixed order: thread-strided partials, warp
// butterfly, then warp 0 adds the 32 warp sums in order.
__device__ __forceinline__ double block_sum_f64(double v, double* red) {
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double s = 0.0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
    return s;
}

__global__ void __launch_bounds__(1024) token_weights_kernel(const float* __restrict__ entropy,
                                                             const uint8_t* __restrict__ is_visual, int T,
                                                             float delta, float eps, float* __restrict__ token_w,
                                                             float* __restrict__ r_v) {
    __shared__ double red[32];
    pdl_wait();
    pdl_trigger();
    double s = 0.0, nv = 0.0;
    for (int t = threadIdx.x; t < T; t += blockDim.x)
        if (is_visual[t]) {
            s += static_cast<double>(entropy[t]);
            nv += 1.0;
        }
    s = block_sum_f64(s, red);
    nv = block_sum_f64(nv, red);
    const double mu = nv > 0.0 ? s / nv : 0.0;
    double var = 0.0;
    for (int t = threadIdx.x; t < T; t += blockDim.x)
        if (is_visual[t]) {
            const double d = static_cast<double>(entropy[t]) - mu;
            var += d * d;
        }
    var = block_sum_f64(var, red);
    const double sigma = nv > 0.0 ? sqrt(var / nv) : 0.0;
    // the z-score's scale once in double; each token's sigmoid in fp32
    const float inv = static_cast<float>(1.0 / (sigma + static_cast<double>(eps)));
    const float muf = static_cast<float>(mu);
    double wv = 0.0, wall = 0.0;
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        float w = 1.0f;
        if (is_visual[t]) {
            const float ht = (entropy[t] - muf) * inv;
            w = 1.0f / (1.0f + expf(delta * ht));
            wv += static_cast<double>(w);
        }
        wall += static_cast<double>(w);
        token_w[t] = w;
    }
    wv = block_sum_f64(wv, red);
    wall = block_sum_f64(wall, red);
    if (threadIdx.x == 0 && r_v != nullptr) *r_v = static_cast<float>(wall > 0.0 ? wv / wall : 0.0);
}

cudaError_t launch_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                                 float eps, float* entropy, float* token_w, float* r_v, moe_dev_status* st,
                                 cudaStream_t s) {
    const dim3 grid((T + 7) / 8);
    cudaError_t e = (x_dtype == MOE_DTYPE_BF16)
                        ? launch_pdl(token_entropy_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                                     static_cast<const __nv_bfloat16*>(x), T, H, entropy, st)
                        : launch_pdl(token_entropy_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(x),
                                     T, H, entropy, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(token_weights_kernel, dim3(1), dim3(1024), 0, s, static_cast<const float*>(entropy), is_visual,
                      T, delta, eps, token_w, r_v);
}

}  // namespace moe
