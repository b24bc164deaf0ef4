// routing.cuh -- the small-batch router tile, per-token ranking (fp32 softmax
// gate, top-R by logit) and the SERE reroute of one token's secondary slots,
// each done by one warp.  Shared by the routing kernels and the fused decode
// routing + dispatch kernel, so that both give bit-identical results.
//
// Gate and ranking: "MACS: Modality-Aware Capacity Scaling for Efficient
// Multimodal MoE Inference", sec. 3.1, Eq. (1).  SERE: Xiaohongshu
// multi-image QA inference article, sec. 4.1-4.2.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Router logits of experts j0 .. j0+EPC-1 for tokens t0 .. t0+3 by a CTA of
// 128 * EPC threads: four warps per expert (one per quarter of H), four
// tokens per warp, the lanes split the quarter (4 consecutive elements each,
// 16-byte weight loads); a fixed xor-butterfly and a fixed-order sum of the
// quarters reduce the partial sums.  part: shared [4 * EPC][4].
// U strips of 128 elements are loaded per batch (all loads of a batch issued
// before any FMA; x is kept as loaded and widened at the FMA); U changes only
// how many loads are in flight, never the order of the FMAs.  The router
// weight is read with an L2 evict-last hint: it is read again every step and
// stays resident while expert weights stream through the L2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float4 ld_f4_keep(const float* p, uint64_t pol) {
    float4 v;
    asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

template <typename XT>
struct XRaw;
template <>
struct XRaw<float> {
    using type = float4;
    static __device__ __forceinline__ type load(const float* p) { return *reinterpret_cast<const float4*>(p); }
    static __device__ __forceinline__ float at(const type& r, int q) {
        return q == 0 ? r.x : q == 1 ? r.y : q == 2 ? r.z : r.w;
    }
    static __device__ __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct XRaw<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ type load(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
    static __device__ __forceinline__ float at(const type& r, int q) {
        const uint32_t u = (q < 2) ? r.x : r.y;
        return __uint_as_float((q & 1) ? (u & 0xffff0000u) : (u << 16));
    }
    static __device__ __forceinline__ type zero() { return make_uint2(0u, 0u); }
};

// Runs nothing; the default step between a router tile's first weight
// prefetches and the rest of it.
struct NoStep {
    __device__ __forceinline__ void operator()() const {}
};

__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

// `mid` is called by every thread of the CTA after the thread's first batch
// of W_r lines has been requested into the L1 and before any x is read: a
// kernel launched as a programmatic dependent passes its dependency wait
// here, since W_r is not written by the launch it waits for, and the first
// weight round trip then overlaps the end of that launch.
template <typename XT, int EPC, int U = 4, typename Mid = NoStep>
__device__ __forceinline__ void router_tile(const XT* __restrict__ x, const float* __restrict__ w, int T, int H,
                                            int N, int j0, int t0, float* __restrict__ logits, float (*part)[4],
                                            Mid mid = Mid()) {
    using XR = XRaw<XT>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = j0 + (warp >> 2);
    const int hq = ((H >> 2) + 127) / 128 * 128;
    const int hbeg = min((warp & 3) * hq, H), hend = min(hbeg + hq, H);
    if (j < N) {
        const float* wr = w + static_cast<size_t>(j) * H;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int h = hbeg + lane * 4 + 128 * u;
            if (h < hend) prefetch_l1(wr + h);
        }
    }
    mid();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (j < N) {
        const uint64_t pol = l2_evict_last_policy();
        const float* wr = w + static_cast<size_t>(j) * H;
        for (int hb = hbeg + lane * 4; hb < hend; hb += 128 * U) {
            float4 wv[U];
            typename XR::type xv[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int h = hb + 128 * u;
                wv[u] = (h < hend) ? ld_f4_keep(wr + h, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int tt = 0; tt < 4; ++tt)
                    xv[u][tt] = (h < hend && t0 + tt < T) ? XR::load(x + static_cast<size_t>(t0 + tt) * H + h)
                                                         : XR::zero();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float wq[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
                for (int tt = 0; tt < 4; ++tt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[tt] = fmaf(XR::at(xv[u][tt], q), wq[q], acc[tt]);
            }
        }
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc[tt] += __shfl_xor_sync(kFull, acc[tt], off);
        }
    }
    if (lane < 4) part[warp][lane] = (lane == 0) ? acc[0] : (lane == 1) ? acc[1] : (lane == 2) ? acc[2] : acc[3];
    __syncthreads();
    if (threadIdx.x < 4 * EPC) {
        const int jl = threadIdx.x >> 2, tt = threadIdx.x & 3;
        const int jj = j0 + jl;
        if (jj < N && t0 + tt < T)
            logits[static_cast<size_t>(t0 + tt) * N + jj] =
                (part[4 * jl][tt] + part[4 * jl + 1][tt]) + (part[4 * jl + 2][tt] + part[4 * jl + 3][tt]);
    }
}

// ---------------------------------------------------------------------------
// Ranking of one token by one warp.  Lane l holds experts j = l + 32 i for
// i < PL (PL = ceil(N/32), a compile-time bound).
// Gate: m = max; e_j = exp_gate(l_j - m); Z = per-lane sums in increasing j,
// then xor butterfly 16, 8, 4, 2, 1; g_j = e_j / Z (IEEE division).
// Ranking: R rounds of a warp arg-best under (logit desc, id asc), each one
// unsigned max of order-preserving keys (redux.sync) and a min over the ids
// holding that key.  On return lane r < R holds (id, gate) of rank r.
// ---------------------------------------------------------------------------
constexpr int kMaxPerLane = MOE_MAX_EXPERTS / 32;

// Unsigned key with the order of the float (all zeros rank as +0; NaN excluded).
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// kCoherent: read the logits with L1-bypassing loads (logits written by other
// CTAs of the same grid).
template <int PL, bool kCoherent = false>
__device__ __forceinline__ bool rank_token(const float* __restrict__ lrow, int N, int R, int k, bool renorm,
                                           int& my_id, float& my_gate) {
    const int lane = threadIdx.x & 31;
    float lv[PL], ev[PL];
    uint32_t kv[PL];
    bool finite = true;
    uint32_t lmax = 0u;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int j = lane + 32 * i;
        lv[i] = (j < N) ? (kCoherent ? __ldcg(lrow + j) : lrow[j]) : 0.f;
        if (j < N && !isfinite(lv[i])) finite = false;
        kv[i] = (j < N) ? order_key(lv[i]) : 0u;   // every finite logit has a key > 0
        lmax = max(lmax, kv[i]);
    }
    const bool all_finite = __all_sync(kFull, finite);
    const float m = key_value(__reduce_max_sync(kFull, lmax));
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int j = lane + 32 * i;
        ev[i] = (j < N) ? exp_gate(__fsub_rn(lv[i], m)) : 0.f;
        if (j < N) part = __fadd_rn(part, ev[i]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(kFull, part, off));
    const float Z = part;
    unsigned taken = 0u;
    my_id = -1;
    for (int r = 0; r < R; ++r) {
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            if (!(taken >> i & 1u) && kv[i] > bk) {   // strict: the lower id wins within the lane
                bk = kv[i];
                bj = lane + 32 * i;
            }
        }
        const uint32_t mk = __reduce_max_sync(kFull, bk);
        const uint32_t cand = (bk == mk && bk != 0u) ? static_cast<uint32_t>(bj) : 0xffffffffu;
        const int jsel = static_cast<int>(__reduce_min_sync(kFull, cand));
        if ((jsel & 31) == lane) {
#pragma unroll
            for (int q = 0; q < PL; ++q)
                if (q == (jsel >> 5)) taken |= 1u << q;
        }
        if (lane == r) my_id = jsel;
    }
    // each lane r < R fetches e of its expert from the owning lane, then divides
    const int mine = my_id >= 0 ? my_id : 0;
    float e_mine = 0.f;
#pragma unroll
    for (int q = 0; q < PL; ++q) {
        const float v = __shfl_sync(kFull, ev[q], mine & 31);
        if (q == (mine >> 5)) e_mine = v;
    }
    my_gate = (lane < R) ? __fdiv_rn(e_mine, Z) : 0.f;
    if (renorm) {
        float s = 0.f;
        for (int r = 0; r < k; ++r) s = __fadd_rn(s, __shfl_sync(kFull, my_gate, r));
        if (lane < k) my_gate = __fdiv_rn(my_gate, s);
    }
    return all_finite;
}

// ---------------------------------------------------------------------------
// SERE reroute of one token's secondary slots by one warp.  Lane r < k holds
// slot r as (id, gate).  P is the primary-union bitmap in shared memory.
// stats: [3] moved, [4] merged, [5] kept-protected, [6] kept-dissimilar.
// ---------------------------------------------------------------------------
template <int PL>
__device__ __forceinline__ void sere_token(int N, int k, int kp, float rho, const float* __restrict__ sim,
                                           const uint8_t* __restrict__ protect, const uint32_t* Pbits,
                                           int& my_id, float& my_gate, int* sstats) {
    const int lane = threadIdx.x & 31;
    for (int r = kp; r < k; ++r) {
        const int s = __shfl_sync(kFull, my_id, r);
        if (s < 0) continue;
        if (Pbits[s >> 5] >> (s & 31) & 1u) continue;
        // the protect bit is consulted once, only for a source about to move
        if (protect != nullptr && protect[s] != 0) {
            if (lane == 0) atomicAdd(&sstats[5], 1);
            continue;
        }
        const float* srow = sim + static_cast<size_t>(s) * N;
        uint32_t bk = 0u;
        int bp = 0;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int p = lane + 32 * i;
            if (p < N && (Pbits[p >> 5] >> (p & 31) & 1u)) {
                const uint32_t key = order_key(srow[p]);
                if (key > bk) {
                    bk = key;
                    bp = p;
                }
            }
        }
        const uint32_t mk = __reduce_max_sync(kFull, bk);
        const uint32_t cand = (bk == mk && bk != 0u) ? static_cast<uint32_t>(bp) : 0xffffffffu;
        const int pbest = static_cast<int>(__reduce_min_sync(kFull, cand));
        if (mk != 0u && key_value(mk) > rho) {
            const unsigned holder = __ballot_sync(kFull, lane < k && my_id == pbest);
            const float gr = __shfl_sync(kFull, my_gate, r);
            if (holder != 0u) {
                const int q = __ffs(holder) - 1;
                if (lane == q) my_gate = __fadd_rn(my_gate, gr);
                if (lane == r) {
                    my_id = -1;
                    my_gate = 0.f;
                }
                if (lane == 0) atomicAdd(&sstats[4], 1);
            } else {
                if (lane == r) my_id = pbest;
                if (lane == 0) atomicAdd(&sstats[3], 1);
            }
        } else if (lane == 0) {
            atomicAdd(&sstats[6], 1);
        }
    }
}

}  // namespace moe
