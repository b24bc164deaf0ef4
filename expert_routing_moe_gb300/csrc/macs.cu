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
// Kernel 1 also leaves per-CTA partials (count, sum, sum of squares of the
// visual entropies, in double, in a fixed order) in the workspace.
// Kernel 2: one CTA reduces the partials in a fixed order (so results are
// reproducible bit for bit), then evaluates each token's sigmoid in fp32 and
// R_v.  (One SM doing the whole reduction in double costs about as much as
// the entropies themselves: fp64 throughput per SM is small.)
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

// Per-CTA partial statistics of the visual tokens' entropies (count, sum,
// sum of squares), in double, summed by thread 0 over its 8 tokens in order.
struct EntPart {
    double n, s, s2;
};

template <typename XT>
__global__ void __launch_bounds__(256) token_entropy_kernel(const XT* __restrict__ x, int T, int H,
                                                            const uint8_t* __restrict__ is_visual,
                                                            float* __restrict__ entropy, EntPart* __restrict__ parts,
                                                            moe_dev_status* st) {
    __shared__ float s_h[8];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (lane == 0) s_h[warp] = 0.f;
    if (t < T) {   // warp-uniform
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
            const float hv = logf(Z) - S1 / Z;
            entropy[t] = hv;
            s_h[warp] = hv;
            if (!all_finite) report(st, MOE_DEV_NONFINITE, t);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        EntPart p{0.0, 0.0, 0.0};
        for (int w = 0; w < 8; ++w) {
            const int tw = blockIdx.x * 8 + w;
            if (tw < T && is_visual[tw]) {
                const double h = static_cast<double>(s_h[w]);
                p.n += 1.0;
                p.s += h;
                p.s2 += h * h;
            }
        }
        parts[blockIdx.x] = p;
    }
}

// Sum over the block in double, fixed order: thread-strided partials, warp
// butterfly, then thread 0 adds the warp sums in order and broadcasts (one
// thread doing the 32 adds: fp64 throughput on one SM is small).
__device__ __forceinline__ double block_sum_f64(double v, double* red) {
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
        red[32] = s;
    }
    __syncthreads();
    return red[32];
}

__global__ void __launch_bounds__(1024) token_weights_kernel(const float* __restrict__ entropy,
                                                             const uint8_t* __restrict__ is_visual, int T,
                                                             const EntPart* __restrict__ parts, int nparts,
                                                             float delta, float eps, float* __restrict__ token_w,
                                                             float* __restrict__ r_v) {
    __shared__ double red[33];
    pdl_wait();
    pdl_trigger();
    double nv = 0.0, s = 0.0, s2 = 0.0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
        nv += parts[i].n;
        s += parts[i].s;
        s2 += parts[i].s2;
    }
    nv = block_sum_f64(nv, red);
    s = block_sum_f64(s, red);
    s2 = block_sum_f64(s2, red);
    // population statistics; the one-pass variance in double is exact to far
    // below the fp32 entropies' own rounding at these magnitudes (|H| <= ln D)
    const double mu = nv > 0.0 ? s / nv : 0.0;
    const double sigma = nv > 0.0 ? sqrt(fmax(s2 / nv - mu * mu, 0.0)) : 0.0;
    // the z-score's scale once in double; each token's sigmoid in fp32
    const float inv = static_cast<float>(1.0 / (sigma + static_cast<double>(eps)));
    const float muf = static_cast<float>(mu);
    float wv = 0.f, wall = 0.f;   // per thread at most ceil(T / 1024) terms
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        float w = 1.0f;
        if (is_visual[t]) {
            const float ht = (entropy[t] - muf) * inv;
            w = 1.0f / (1.0f + expf(delta * ht));
            wv += w;
        }
        wall += w;
        token_w[t] = w;
    }
    const double wvs = block_sum_f64(static_cast<double>(wv), red);
    const double walls = block_sum_f64(static_cast<double>(wall), red);
    if (threadIdx.x == 0 && r_v != nullptr) *r_v = static_cast<float>(walls > 0.0 ? wvs / walls : 0.0);
}

size_t token_weights_workspace(int T) { return static_cast<size_t>((T + 7) / 8) * sizeof(EntPart); }

cudaError_t launch_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                                 float eps, float* entropy, float* token_w, float* r_v, void* ws, moe_dev_status* st,
                                 cudaStream_t s) {
    const int nb = (T + 7) / 8;
    EntPart* parts = static_cast<EntPart*>(ws);
    cudaError_t e = (x_dtype == MOE_DTYPE_BF16)
                        ? launch_pdl(token_entropy_kernel<__nv_bfloat16>, dim3(nb), dim3(256), 0, s,
                                     static_cast<const __nv_bfloat16*>(x), T, H, is_visual, entropy, parts, st)
                        : launch_pdl(token_entropy_kernel<float>, dim3(nb), dim3(256), 0, s,
                                     static_cast<const float*>(x), T, H, is_visual, entropy, parts, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(token_weights_kernel, dim3(1), dim3(1024), 0, s, static_cast<const float*>(entropy), is_visual,
                      T, static_cast<const EntPart*>(parts), nb, delta, eps, token_w, r_v);
}

}  // namespace moe
