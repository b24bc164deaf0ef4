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
// Kernel 1: one warp per token.  With m = max z and the exponent taken in
// base 2, u_d = (z_d - m) log2(e) formed by one FMA and e_d = 2^u_d (the
// hardware's approximate exponential: its error is far below the entropy's
// fp32 summation error), H = ln Z - ln 2 * (sum e_d u_d) / Z, in a fixed lane
// order with an xor butterfly.  A row of up to 2048 features is read once
// into registers (bf16 rows stay packed, 32 registers a lane; their maximum
// is taken on the packed pairs) and both passes run from there.  A
// non-finite feature always makes H NaN (NaN propagates, +inf gives
// inf - inf, -inf gives 0 * -inf), so H itself is the finiteness test.
// Each CTA leaves the count, sum and sum of squares of its visual tokens'
// entropies as 64-bit fixed-point integers (2^-32 and 2^-24 units).
// Kernel 2: one thread per token over ceil(T / 256) CTAs.  Every CTA adds up
// the kernel-1 partials itself; integer sums do not depend on their order,
// so every CTA holds the same statistics.  n^2 times the variance is formed
// exactly from them in 128-bit integers (n sum h^2 - (sum h)^2, no
// cancellation), then mean and 1/(sigma + eps) in fp32 by one thread: double
// precision is slow on this part and sits on the critical path here.  Each
// thread evaluates its token's sigmoid in fp32; the CTA's (visual, total)
// weight sums are again fixed-point integers (2^-32 units), which the last
// CTA to finish (a ticket that kernel 1 clears) adds up for R_v.  So the
// results are reproducible bit for bit.
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

// Per-CTA partial statistics of the visual tokens' entropies: count, sum
// (2^-32 units) and sum of squares (2^-24 units) as integers.  Entropies lie
// in [0, ln D], so with T <= 2^24 tokens neither sum can overflow.
struct EntPart {
    long long n, s1, s2;
};
constexpr float kEntScale1 = 4294967296.0f;   // 2^32
constexpr float kEntScale2 = 16777216.0f;     // 2^24
constexpr float kWScale = 4294967296.0f;      // 2^32, weights in [0, 1]

// h*h in 2^-24 units, from its exact two-term fp32 split (hi + lo = h*h).
__device__ __forceinline__ long long sq_fixed(float h) {
    const float hi = h * h;
    const float lo = fmaf(h, h, -hi);
    return __float2ll_rn(hi * kEntScale2) + __float2ll_rn(lo * kEntScale2);
}

// Chunks of 8 features per lane that a register-cached row holds (H <= 2048).
constexpr int kEntRegChunks = 8;

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

constexpr float kL2E = 0x1.715476p+0f;   // log2(e), nearest fp32
constexpr float kLn2 = 0x1.62e430p-1f;   // ln(2), nearest fp32

// 2^u, the approximate hardware exponential (subnormal results flushed to 0;
// 2^-inf = 0, NaN stays NaN).
__device__ __forceinline__ float ex2_approx(float u) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(u));
    return y;
}

// Elementwise maximum of two packed bf16 pairs.
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __nv_bfloat162 r = __hmax2(x, y);
    uint32_t o;
    memcpy(&o, &r, 4);
    return o;
}

// The terms of one feature: e = 2^u with u = z log2(e) - ml, ml = m log2(e).
__device__ __forceinline__ void ent_term(float z, float ml, float& Z, float& S1) {
    const float u = fmaf(z, kL2E, -ml);
    const float e = ex2_approx(u);
    Z += e;
    S1 = fmaf(e, u, S1);
}

// Max, then Z = sum e and S1 = sum e * u (base-2 exponents), over one lane's
// chunks of a row.
template <typename XT, bool CACHED>
__device__ __forceinline__ void entropy_lane_sums(const XT* row, int H, int lane, float& m, float& Z, float& S1) {
    if constexpr (CACHED && sizeof(XT) == 2) {
        // bf16 row kept packed: 8 x 16 bytes per lane, unpacked in the second pass
        uint4 q[kEntRegChunks];
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            const int h = lane * 8 + c * 256;
            q[c] = (h < H) ? *reinterpret_cast<const uint4*>(row + h) : make_uint4(0u, 0u, 0u, 0u);
        }
        uint32_t mx = 0xff80ff80u;   // (-inf, -inf)
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            if (lane * 8 + c * 256 < H) {
                mx = bf2_max(mx, bf2_max(bf2_max(q[c].x, q[c].y), bf2_max(q[c].z, q[c].w)));
            }
        }
        m = fmaxf(bf_lo(mx), bf_hi(mx));
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
        const float ml = m * kL2E;
        Z = 0.f;
        S1 = 0.f;
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            if (lane * 8 + c * 256 < H) {
                const uint32_t u[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ent_term(bf_lo(u[j]), ml, Z, S1);
                    ent_term(bf_hi(u[j]), ml, Z, S1);
                }
            }
        }
    } else if constexpr (CACHED) {
        float v[kEntRegChunks][8];
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            const int h = lane * 8 + c * 256;
            if (h < H) {
                load8(row + h, v[c]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[c][j] = -INFINITY;
            }
        }
        m = -INFINITY;
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            if (lane * 8 + c * 256 < H) {
#pragma unroll
                for (int j = 0; j < 8; ++j) m = fmaxf(m, v[c][j]);
            }
        }
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
        const float ml = m * kL2E;
        Z = 0.f;
        S1 = 0.f;
#pragma unroll
        for (int c = 0; c < kEntRegChunks; ++c) {
            if (lane * 8 + c * 256 < H) {
#pragma unroll
                for (int j = 0; j < 8; ++j) ent_term(v[c][j], ml, Z, S1);
            }
        }
    } else {
        m = -INFINITY;
        for (int h = lane * 8; h < H; h += 256) {
            float v[8];
            load8(row + h, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, v[j]);
        }
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
        const float ml = m * kL2E;
        Z = 0.f;
        S1 = 0.f;
        for (int h = lane * 8; h < H; h += 256) {
            float v[8];
            load8(row + h, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) ent_term(v[j], ml, Z, S1);
        }
    }
}

// An unsigned 128-bit integer to the nearest fp32 or a neighbour (two
// conversions and one fused rounding: a few ulp).
__device__ __forceinline__ float u128_to_float(unsigned __int128 v) {
    const float hi = static_cast<float>(static_cast<unsigned long long>(v >> 64));
    const float lo = static_cast<float>(static_cast<unsigned long long>(v));
    return fmaf(hi, 18446744073709551616.0f, lo);   // hi * 2^64 + lo
}

// Sums of the weights of one CTA of kernel 2 (visual, all), 2^-32 units.
struct WPart {
    long long wv, wall;
};

// Sum of NV int64 values over the block (any order gives the same result);
// every thread gets the totals.  red: [NV][33].
template <int NV>
__device__ __forceinline__ void block_sum_i64(long long (&v)[NV], long long (*red)[33]) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
        for (int off = 16; off >= 1; off >>= 1) v[i] += __shfl_xor_sync(kFull, v[i], off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) red[i][threadIdx.x >> 5] = v[i];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int nw = static_cast<int>(blockDim.x >> 5);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            long long t = static_cast<int>(threadIdx.x) < nw ? red[i][threadIdx.x] : 0;
            for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(kFull, t, off);
            if (threadIdx.x == 0) red[i][32] = t;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = red[i][32];
}

template <typename XT, bool CACHED>
__global__ void __launch_bounds__(256) token_entropy_kernel(const XT* __restrict__ x, int T, int H,
                                                            const uint8_t* __restrict__ is_visual,
                                                            float* __restrict__ entropy, EntPart* __restrict__ parts,
                                                            int* __restrict__ ticket, moe_dev_status* st) {
    __shared__ float s_h[8];
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;   // kernel 2's ticket, cleared for this call
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (lane == 0) s_h[warp] = 0.f;
    if (t < T) {   // warp-uniform
        const XT* row = x + static_cast<size_t>(t) * H;
        float m, Z, S1;
        entropy_lane_sums<XT, CACHED>(row, H, lane, m, Z, S1);
        for (int off = 16; off >= 1; off >>= 1) {
            Z += __shfl_xor_sync(kFull, Z, off);
            S1 += __shfl_xor_sync(kFull, S1, off);
        }
        if (lane == 0) {
            const float hv = logf(Z) - kLn2 * (S1 / Z);
            entropy[t] = hv;
            s_h[warp] = hv;
            if (!isfinite(hv)) report(st, MOE_DEV_NONFINITE, t);
        }
    }
    __syncthreads();
    if (warp == 0) {
        // lanes 0..7: this CTA's tokens as fixed-point terms, summed with integer shuffles
        const int tw = blockIdx.x * 8 + lane;
        const bool v = lane < 8 && tw < T && is_visual[tw] != 0;
        const float h = v ? s_h[lane] : 0.f;
        long long n = v ? 1 : 0, q1 = v ? __float2ll_rn(h * kEntScale1) : 0, q2 = v ? sq_fixed(h) : 0;
        for (int off = 4; off >= 1; off >>= 1) {
            n += __shfl_xor_sync(kFull, n, off);
            q1 += __shfl_xor_sync(kFull, q1, off);
            q2 += __shfl_xor_sync(kFull, q2, off);
        }
        if (lane == 0) parts[blockIdx.x] = EntPart{n, q1, q2};
    }
}

__global__ void __launch_bounds__(256) token_weights_kernel(const float* __restrict__ entropy,
                                                            const uint8_t* __restrict__ is_visual, int T,
                                                            const EntPart* __restrict__ parts, int nparts,
                                                            float delta, float eps, float* __restrict__ token_w,
                                                            WPart* __restrict__ wparts, int* __restrict__ ticket,
                                                            float* __restrict__ r_v) {
    __shared__ long long red[3][33];
    __shared__ float s_mu, s_inv;
    __shared__ bool s_last;
    pdl_wait();
    pdl_trigger();
    // this thread's token, loaded before the statistics are reduced
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const bool vis_t = t < T && is_visual[t] != 0;
    const float ent_t = vis_t ? entropy[t] : 0.f;
    long long st3[3] = {0, 0, 0};   // count, sum, sum of squares (fixed point)
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
        const EntPart p = parts[i];
        st3[0] += p.n;
        st3[1] += p.s1;
        st3[2] += p.s2;
    }
    block_sum_i64<3>(st3, red);
    // population statistics by one thread, without double precision (slow on
    // this part): n^2 * var * 2^64 = n * S2 * 2^40 - S1^2 exactly in 128-bit
    // integers (entropies in 2^-32 units, squares in 2^-24), then fp32.
    if (threadIdx.x == 0) {
        const long long n = st3[0];
        float mu = 0.f, sigma = 0.f;
        if (n > 0) {
            const float nq = static_cast<float>(n) * 4294967296.0f;   // n * 2^32, exact for n <= 2^24
            mu = static_cast<float>(st3[1]) / nq;
            const __int128 num = (static_cast<__int128>(n) * st3[2] << 40) - static_cast<__int128>(st3[1]) * st3[1];
            sigma = num > 0 ? sqrtf(u128_to_float(static_cast<unsigned __int128>(num))) / nq : 0.f;
        }
        s_mu = mu;
        s_inv = 1.0f / (sigma + eps);
    }
    __syncthreads();
    const float inv = s_inv, muf = s_mu;
    float w = 0.f, wv = 0.f;
    if (t < T) {
        w = 1.0f;
        if (vis_t) {
            const float ht = (ent_t - muf) * inv;
            w = 1.0f / (1.0f + expf(delta * ht));
            wv = w;
        }
        token_w[t] = w;
    }
    if (r_v == nullptr) return;   // uniform over the grid
    long long ws2[2] = {__float2ll_rn(wv * kWScale), __float2ll_rn(w * kWScale)};
    block_sum_i64<2>(ws2, red);
    if (threadIdx.x == 0) {
        wparts[blockIdx.x] = WPart{ws2[0], ws2[1]};
        __threadfence();
        s_last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (!s_last) return;   // uniform over the block
    __threadfence();
    long long tot[2] = {0, 0};
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) {
        tot[0] += __ldcg(&wparts[i].wv);
        tot[1] += __ldcg(&wparts[i].wall);
    }
    block_sum_i64<2>(tot, red);
    if (threadIdx.x == 0) {
        *r_v = tot[1] > 0 ? static_cast<float>(tot[0]) / static_cast<float>(tot[1]) : 0.f;
        *ticket = 0;
    }
}

// Workspace: kernel-1 partials, kernel-2 partials, the ticket.
static size_t ent_parts_bytes(int T) { return static_cast<size_t>((T + 7) / 8) * sizeof(EntPart); }
static size_t w_parts_bytes(int T) { return static_cast<size_t>((T + 255) / 256) * sizeof(WPart); }

size_t token_weights_workspace(int T) { return ent_parts_bytes(T) + w_parts_bytes(T) + 16; }

cudaError_t launch_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                                 float eps, float* entropy, float* token_w, float* r_v, void* ws, moe_dev_status* st,
                                 cudaStream_t s) {
    const int nb = (T + 7) / 8;
    EntPart* parts = static_cast<EntPart*>(ws);
    WPart* wparts = reinterpret_cast<WPart*>(static_cast<char*>(ws) + ent_parts_bytes(T));
    int* ticket = reinterpret_cast<int*>(static_cast<char*>(ws) + ent_parts_bytes(T) + w_parts_bytes(T));
    const bool cached = H <= kEntRegChunks * 256;
    cudaError_t e;
    if (x_dtype == MOE_DTYPE_BF16) {
        const auto* xb = static_cast<const __nv_bfloat16*>(x);
        e = cached ? launch_pdl(token_entropy_kernel<__nv_bfloat16, true>, dim3(nb), dim3(256), 0, s, xb, T, H,
                                is_visual, entropy, parts, ticket, st)
                   : launch_pdl(token_entropy_kernel<__nv_bfloat16, false>, dim3(nb), dim3(256), 0, s, xb, T, H,
                                is_visual, entropy, parts, ticket, st);
    } else {
        const auto* xf = static_cast<const float*>(x);
        e = cached ? launch_pdl(token_entropy_kernel<float, true>, dim3(nb), dim3(256), 0, s, xf, T, H, is_visual,
                                entropy, parts, ticket, st)
                   : launch_pdl(token_entropy_kernel<float, false>, dim3(nb), dim3(256), 0, s, xf, T, H, is_visual,
                                entropy, parts, ticket, st);
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(token_weights_kernel, dim3((T + 255) / 256), dim3(256), 0, s, static_cast<const float*>(entropy),
                      is_visual, T, static_cast<const EntPart*>(parts), nb, delta, eps, token_w, wparts, ticket, r_v);
}

}  // namespace moe
