// router.cu -- router GEMM, fp32 softmax gate + top-R ranking, and the SERE
// batch reroute fused into the ranking kernel.
//
// Router and gate: "MACS: Modality-Aware Capacity Scaling for Efficient
// Multimodal MoE Inference", sec. 3.1, Eq. (1).
// SERE: Xiaohongshu multi-image QA inference article, sec. 4.1 (primary
// union as the shared candidate set, most-similar primary above rho) and
// sec. 4.2 (one fused operator, protection of source experts only).
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

// ---------------------------------------------------------------------------
// Router GEMM, small batches: one warp per expert, four tokens per warp, the
// lanes split H (4 consecutive elements each, 16-byte weight loads) and a
// fixed xor-butterfly reduces the partial sums.  Grid (ceil(N/8), ceil(T/4)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
    uint2 q = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
}

template <typename XT>
__global__ void __launch_bounds__(256) router_warp_kernel(const XT* __restrict__ x, const float* __restrict__ w,
                                                          int T, int H, int N, float* __restrict__ logits) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = blockIdx.x * 8 + warp;
    const int t0 = blockIdx.y * 4;
    if (j >= N) return;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float* wr = w + static_cast<size_t>(j) * H;
    for (int h = lane * 4; h < H; h += 128) {
        float wv[4];
        load4(wr + h, wv);
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
            if (t0 + tt < T) {
                float xv[4];
                load4(x + static_cast<size_t>(t0 + tt) * H + h, xv);
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[tt] = fmaf(xv[q], wv[q], acc[tt]);
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc[tt] += __shfl_xor_sync(kFull, acc[tt], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int tt = 0; tt < 4; ++tt)
            if (t0 + tt < T) logits[static_cast<size_t>(t0 + tt) * N + j] = acc[tt];
    }
}

// ---------------------------------------------------------------------------
// Router GEMM, large batches: 64 tokens x 64 experts per CTA, 256 threads,
// 4x4 outputs per thread, K staged through shared memory 32 at a time.
// ---------------------------------------------------------------------------
template <typename XT>
__global__ void __launch_bounds__(256) router_tiled_kernel(const XT* __restrict__ x, const float* __restrict__ w,
                                                           int T, int H, int N, float* __restrict__ logits) {
    constexpr int TM = 64, TN = 64, TK = 32;
    __shared__ float xs[TK][TM + 4];
    __shared__ float ws[TK][TN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int tb = blockIdx.y * TM, jb = blockIdx.x * TN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < H; k0 += TK) {
        // 64 rows x 32 k for each operand: 2048 values, 8 per thread
        for (int e = tid; e < TM * TK; e += 256) {
            const int r = e / TK, c = e % TK;
            const int t = tb + r, h = k0 + c;
            float v = 0.f;
            if (t < T && h < H) {
                if constexpr (sizeof(XT) == 2) {
                    v = __bfloat162float(x[static_cast<size_t>(t) * H + h]);
                } else {
                    v = x[static_cast<size_t>(t) * H + h];
                }
            }
            xs[c][r] = v;
            const int j = jb + r;
            ws[c][r] = (j < N && h < H) ? w[static_cast<size_t>(j) * H + h] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i) b[i] = ws[kk][tx * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = tb + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = jb + tx * 4 + jj;
            if (j < N) logits[static_cast<size_t>(t) * N + j] = acc[i][jj];
        }
    }
}

cudaError_t launch_router(const void* x, int x_dtype, const float* w_router, int T, int H, int N, float* logits,
                          cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (T <= 256) {
        dim3 grid((N + 7) / 8, (T + 3) / 4);
        if (x_dtype == MOE_DTYPE_BF16)
            router_warp_kernel<__nv_bfloat16>
                <<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), w_router, T, H, N, logits);
        else
            router_warp_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x), w_router, T, H, N, logits);
    } else {
        dim3 grid((N + 63) / 64, (T + 63) / 64);
        if (x_dtype == MOE_DTYPE_BF16)
            router_tiled_kernel<__nv_bfloat16>
                <<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), w_router, T, H, N, logits);
        else
            router_tiled_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x), w_router, T, H, N, logits);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Ranking of one token by one warp.  Lane l holds experts j = l + 32 i.
// Gate: m = max; e_j = exp_gate(l_j - m); Z = per-lane sums in increasing j,
// then xor butterfly 16, 8, 4, 2, 1; g_j = e_j / Z (IEEE division).
// Ranking: R rounds of warp arg-best under (logit desc, id asc).
// On return lane r < R holds (id, gate) of rank r.
// ---------------------------------------------------------------------------
constexpr int kMaxPerLane = MOE_MAX_EXPERTS / 32;

__device__ __forceinline__ bool rank_token(const float* __restrict__ lrow, int N, int R, int k, bool renorm,
                                           int& my_id, float& my_gate) {
    const int lane = threadIdx.x & 31;
    float lv[kMaxPerLane], ev[kMaxPerLane];
    bool finite = true;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        lv[i] = (j < N) ? lrow[j] : 0.f;
        if (j < N && !isfinite(lv[i])) finite = false;
    }
    const bool all_finite = __all_sync(kFull, finite);
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i < N) m = fmaxf(m, lv[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        ev[i] = (j < N) ? exp_gate(__fsub_rn(lv[i], m)) : 0.f;
        if (j < N) part = __fadd_rn(part, ev[i]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(kFull, part, off));
    const float Z = part;
    unsigned taken = 0u;
    my_id = -1;
    my_gate = 0.f;
    for (int r = 0; r < R; ++r) {
        float bv = 0.f;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int j = lane + 32 * i;
            if (j < N && !(taken >> i & 1u) && (bi < 0 || ranks_before(lv[i], j, bv, bi))) {
                bv = lv[i];
                bi = j;
            }
        }
        warp_best(bv, bi);
        float g = 0.f;
        if ((bi & 31) == lane) {
            const int i = bi >> 5;
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q)
                if (q == i) {
                    taken |= 1u << q;
                    g = __fdiv_rn(ev[q], Z);
                }
        }
        g = __shfl_sync(kFull, g, bi & 31);
        if (lane == r) {
            my_id = bi;
            my_gate = g;
        }
    }
    if (renorm) {
        float s = 0.f;
        for (int r = 0; r < k; ++r) s = __fadd_rn(s, __shfl_sync(kFull, my_gate, r));
        if (lane < k) my_gate = __fdiv_rn(my_gate, s);
    }
    return all_finite;
}

__global__ void __launch_bounds__(256) rank_kernel(const float* __restrict__ logits, int T, int N, int R, int k,
                                                   int renorm, int32_t* __restrict__ ids,
                                                   float* __restrict__ gates, moe_dev_status* st) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int id;
    float g;
    const bool ok = rank_token(logits + static_cast<size_t>(t) * N, N, R, k, renorm != 0, id, g);
    if (!ok && lane == 0) report(st, MOE_DEV_NONFINITE, t);
    if (lane < R) {
        ids[static_cast<size_t>(t) * R + lane] = id;
        gates[static_cast<size_t>(t) * R + lane] = g;
    }
}

cudaError_t launch_rank(const float* logits, int T, int N, int R, int k, bool renorm, int32_t* ids, float* gates,
                        moe_dev_status* st, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    rank_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, N, R, k, renorm ? 1 : 0, ids, gates, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SERE reroute of one token's secondary slots by one warp.  Lane r < k holds
// slot r as (id, gate).  P is the primary-union bitmap in shared memory.
// stats: [3] moved, [4] merged, [5] kept-protected, [6] kept-dissimilar.
// ---------------------------------------------------------------------------
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
        float bv = 0.f;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int p = lane + 32 * i;
            if (p < N && (Pbits[p >> 5] >> (p & 31) & 1u)) {
                const float v = srow[p];
                if (bi < 0 || ranks_before(v, p, bv, bi)) {
                    bv = v;
                    bi = p;
                }
            }
        }
        warp_best(bv, bi);
        if (bi >= 0 && bv > rho) {
            const unsigned holder = __ballot_sync(kFull, lane < k && my_id == bi);
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
                if (lane == r) my_id = bi;
                if (lane == 0) atomicAdd(&sstats[3], 1);
            }
        } else if (lane == 0) {
            atomicAdd(&sstats[6], 1);
        }
    }
}

// One CTA of 1024 threads handles the whole batch: (optionally) rank every
// token, build the primary union P and the before-union, reroute, build the
// after-union, publish stats.  No host synchronisation, no extra sort.
__global__ void __launch_bounds__(1024) rank_sere_kernel(const float* __restrict__ logits, int do_rank, int T,
                                                         int N, int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ gates, int ld, int kp, float rho,
                                                         const float* __restrict__ sim,
                                                         const uint8_t* __restrict__ protect,
                                                         uint32_t* __restrict__ union_bitmap,
                                                         int32_t* __restrict__ stats, moe_dev_status* st) {
    __shared__ uint32_t Pbits[kMaxPerLane], Ubefore[kMaxPerLane], Uafter[kMaxPerLane];
    __shared__ int sstats[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < kMaxPerLane) {
        Pbits[threadIdx.x] = 0u;
        Ubefore[threadIdx.x] = 0u;
        Uafter[threadIdx.x] = 0u;
    }
    if (threadIdx.x < 8) sstats[threadIdx.x] = 0;
    __syncthreads();
    for (int t = warp; t < T; t += 32) {
        int id = -1;
        float g = 0.f;
        if (do_rank) {
            const bool ok = rank_token(logits + static_cast<size_t>(t) * N, N, k, k, renorm != 0, id, g);
            if (!ok && lane == 0) report(st, MOE_DEV_NONFINITE, t);
            if (lane < k) {
                ids[static_cast<size_t>(t) * ld + lane] = id;
                gates[static_cast<size_t>(t) * ld + lane] = g;
            }
        } else if (lane < k) {
            id = ids[static_cast<size_t>(t) * ld + lane];
        }
        if (lane < k && id >= N) report(st, MOE_DEV_BAD_INDEX, id);
        if (lane < k && id >= 0 && id < N) {
            atomicOr(&Ubefore[id >> 5], 1u << (id & 31));
            if (lane < kp) atomicOr(&Pbits[id >> 5], 1u << (id & 31));
        }
    }
    __syncthreads();
    for (int t = warp; t < T; t += 32) {
        int id = -1;
        float g = 0.f;
        if (lane < k) {
            id = ids[static_cast<size_t>(t) * ld + lane];
            g = gates[static_cast<size_t>(t) * ld + lane];
            if (id >= N) id = -1;
        }
        sere_token(N, k, kp, rho, sim, protect, Pbits, id, g, sstats);
        if (lane < k) {
            ids[static_cast<size_t>(t) * ld + lane] = id;
            gates[static_cast<size_t>(t) * ld + lane] = g;
            if (id >= 0) atomicOr(&Uafter[id >> 5], 1u << (id & 31));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ub = 0, np = 0, ua = 0;
        for (int w = 0; w < kMaxPerLane; ++w) {
            ub += __popc(Ubefore[w]);
            np += __popc(Pbits[w]);
            ua += __popc(Uafter[w]);
        }
        if (stats != nullptr) {
            stats[0] = ub;
            stats[1] = np;
            stats[2] = ua;
            for (int i = 3; i < 7; ++i) stats[i] = sstats[i];
            stats[7] = 0;
        }
    }
    if (union_bitmap != nullptr && threadIdx.x < (N + 31) / 32) union_bitmap[threadIdx.x] = Pbits[threadIdx.x];
}

cudaError_t launch_rank_sere(const float* logits, int T, int N, int k, bool renorm, int32_t* ids, float* gates,
                             const moe_sere_params& p, moe_dev_status* st, cudaStream_t s) {
    rank_sere_kernel<<<1, 1024, 0, s>>>(logits, 1, T, N, k, renorm ? 1 : 0, ids, gates, k, p.k_primary, p.rho,
                                        p.sim, p.protect, p.union_bitmap, p.stats, st);
    return cudaGetLastError();
}

cudaError_t launch_sere(int32_t* ids, float* gates, int ld, int T, int N, int k, const moe_sere_params& p,
                        moe_dev_status* st, cudaStream_t s) {
    rank_sere_kernel<<<1, 1024, 0, s>>>(nullptr, 0, T, N, k, 0, ids, gates, ld, p.k_primary, p.rho, p.sim,
                                        p.protect, p.union_bitmap, p.stats, st);
    return cudaGetLastError();
}

}  // namespace moe
