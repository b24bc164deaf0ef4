// routing.cuh -- per-token ranking (fp32 softmax gate, top-R by logit) and the
// SERE reroute of one token's secondary slots, each done by one warp.  Shared
// by the routing kernels and the fused decode layer kernel.
//
// Gate and ranking: "MACS: Modality-Aware Capacity Scaling for Efficient
// Multimodal MoE Inference", sec. 3.1, Eq. (1).  SERE: Xiaohongshu
// multi-image QA inference article, sec. 4.1-4.2.
#pragma once

#include "common.cuh"

namespace moe {

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

template <int PL>
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
        lv[i] = (j < N) ? lrow[j] : 0.f;
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
