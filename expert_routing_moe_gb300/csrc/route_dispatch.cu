// route_dispatch.cu -- decode routing and dispatch in one launch: the router
// GEMM, the fp32 softmax gate and top-k ranking, the SERE batch reroute and
// the expert-sorted permutation.
//
// Router and gate: "MACS: Modality-Aware Capacity Scaling for Efficient
// Multimodal MoE Inference", sec. 3.1, Eq. (1); SERE: Xiaohongshu multi-image
// QA inference article, sec. 4.1 (primary union, most similar primary above
// rho) and sec. 4.2 (one operator feeding the fused MoE with no host round
// trip, protection of source experts); the permutation orders rows by
// (expert, token), the token sets of "MACS" Eq. (2).
//
// At decode sizes every step after the router GEMM touches a few KB, so
// separate launches cost more than their work, and so does doing all of it on
// one SM (ranking a token is ~600 warp instructions).  The grid is (expert
// tiles of 8) x (token groups of 4); no CTA ever waits for another:
//  1. every CTA computes its tile of router logits (router_tile, the
//     arithmetic of the standalone router kernel);
//  2. the last CTA of each token group (a per-group ticket) ranks the
//     group's tokens, one warp per token, and ORs their primaries and experts
//     into the batch's union bitmaps in the workspace;
//  3. the last group to finish (a second ticket) chooses the SERE target of
//     every source expert that some token holds outside P, once, over the
//     members of P (the similarity staged in shared memory by a bulk copy
//     that every group-ranking CTA issues before it ranks), reroutes each
//     token's movers, and writes the permutation, with the batch's slots held
//     in shared memory throughout.
// On one SM the tail is bound by shared-memory and warp-collective
// throughput, not latency, so it does only the needed work: targets for the
// held sources only, and only the movers of each token.
// Tickets and bitmaps are returned to zero by the CTAs that consumed them, so
// the workspace is zero between calls.  The outputs are bit-identical to
// moe_route followed by the uncapped moe_dispatch_capacity.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "permute.cuh"   // block_count
#include "routing.cuh"

namespace moe {

constexpr int kRdThreads = 1024;   // 32 warps: 8 experts x 4 quarters in the router tile
constexpr int kRdEpc = kRdThreads / 128;
constexpr int kRdStageN = 128;     // the similarity is staged in shared memory up to N = 128 (64 KiB)

// Workspace words (int32): [0] batch ticket, [8, 16) primary union P,
// [16, 24) union before the reroute, [32, 32 + ceil(T/4)) group tickets,
// [96] early flag and [97, 105) early bitmap (published for the decode FFN).
constexpr int kWsTicket = 0, kWsP = 8, kWsUb = 16, kWsGroups = 32, kWsEarly = kRouteDispatchEarlyWord;
static_assert(kWsGroups + kRouteDispatchMaxT / 4 <= kWsEarly, "workspace words");
static_assert(kWsEarly + 1 + kMaxPerLane <= kRouteDispatchWs / 4, "workspace words");

struct RdArgs {
    int T, H, N, k, kp, renorm, stage_sim, publish, spec_max;
    float rho;
    const float* sim;
    const uint8_t* protect;
    uint32_t* union_bitmap;
    int32_t* stats;
    float* logits;
    int32_t* ids;
    float* gates;
    int32_t* counts;
    int32_t* offsets;
    int32_t* row_token;
    float* row_gate;
    int32_t* active;
    int* ws;
};

// Stage 2: rank the tokens of group g (one warp per token) into ids/gates and
// the workspace's union bitmaps.
template <int PL, bool SERE>
__device__ __forceinline__ void rank_group(const RdArgs& a, int g, moe_dev_status* st) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = g * 4 + warp;
    if (warp >= 4 || t >= a.T) return;
    int id;
    float gt;
    const bool ok = rank_token<PL, true>(a.logits + static_cast<size_t>(t) * a.N, a.N, a.k, a.k, a.renorm != 0, id,
                                         gt);
    if (!ok && lane == 0) report(st, MOE_DEV_NONFINITE, t);
    if (lane < a.k) {
        a.ids[static_cast<size_t>(t) * a.k + lane] = id;
        a.gates[static_cast<size_t>(t) * a.k + lane] = gt;
        if ((SERE || a.publish) && id >= 0 && id < a.N) {
            uint32_t* ws = reinterpret_cast<uint32_t*>(a.ws);
            atomicOr(&ws[kWsUb + (id >> 5)], 1u << (id & 31));
            if (SERE && lane < a.kp) atomicOr(&ws[kWsP + (id >> 5)], 1u << (id & 31));
        }
    }
}

// Compacts the set bits of bm[0 .. ceil(N/32)) into list (ascending) with
// one warp; returns the count in lane 0's result.
__device__ __forceinline__ int compact_bits(const uint32_t* bm, int N, int* list) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    for (int w = 0; w < (N + 31) / 32; ++w) {
        const uint32_t b = bm[w];
        if (b >> lane & 1u) list[base + __popc(b & ((1u << lane) - 1u))] = 32 * w + lane;
        base += __popc(b);
    }
    return base;
}

// Exclusive scan of the per-expert row counts over up to 8 warps (N <= 256):
// counts, offsets (with the total at [N]), the active list and start[e].
// Returns the number of active experts (in every thread).
__device__ __forceinline__ int scan_experts_warps(const int* cnt, int N, int32_t* counts, int32_t* offsets,
                                                  int32_t* active, int* start) {
    __shared__ int wsum[MOE_MAX_EXPERTS / 32], wact[MOE_MAX_EXPERTS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, e = threadIdx.x;
    const int nwarps = (N + 31) / 32;
    int c = 0, act = 0, inc = 0, ainc = 0;
    if (warp < nwarps) {
        c = (e < N) ? cnt[e] : 0;
        act = c > 0 ? 1 : 0;
        inc = c;
        ainc = act;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFull, inc, off);
            const int av = __shfl_up_sync(kFull, ainc, off);
            if (lane >= off) {
                inc += v;
                ainc += av;
            }
        }
        if (lane == 31) {
            wsum[warp] = inc;
            wact[warp] = ainc;
        }
    }
    __syncthreads();
    if (e < N) {
        int base = 0, abase = 0;
        for (int w = 0; w < warp; ++w) {
            base += wsum[w];
            abase += wact[w];
        }
        const int o = base + inc - c;
        start[e] = o;
        counts[e] = c;
        offsets[e] = o;
        if (act) active[abase + ainc] = e;   // 1 + (exclusive position)
    }
    int tot = 0, atot = 0;
    for (int w = 0; w < nwarps; ++w) {
        tot += wsum[w];
        atot += wact[w];
    }
    if (threadIdx.x == 0) {
        offsets[N] = tot;
        active[0] = atot;
    }
    return atot;
}

// SERE of one token's secondaries (lane r < k holds slot r as (id, gate)),
// with the target of each source outside P already in tgt/tkey.  The movers
// -- secondaries outside P, not protected, whose target similarity exceeds
// rho -- are taken in rank order, exactly as in sere_token: a mover merges
// into the slot that currently holds its target (a kept slot, or an earlier
// mover that took that target), else it takes the target.  Slots that do not
// move never change, so only the movers are visited.  cnt4 accumulates
// (moved, merged, kept-protected, kept-dissimilar), the same in every lane.
__device__ __forceinline__ void sere_token_movers(int k, int kp, float rho, const uint8_t* protect,
                                                  const uint32_t* Pbits, const int* tgt, const uint32_t* tkey,
                                                  int& my_id, float& my_gate, int (&cnt4)[4]) {
    const int lane = threadIdx.x & 31;
    const int s = my_id;
    bool moving = false, kept_prot = false, kept_dis = false;
    int fin = -1;
    if (lane >= kp && lane < k && s >= 0 && !(Pbits[s >> 5] >> (s & 31) & 1u)) {
        if (protect != nullptr && protect[s] != 0) {
            kept_prot = true;
        } else {
            const uint32_t mk = tkey[s];
            moving = mk != 0u && key_value(mk) > rho;
            kept_dis = !moving;
            fin = tgt[s];
        }
    }
    cnt4[2] += __popc(__ballot_sync(kFull, kept_prot));
    cnt4[3] += __popc(__ballot_sync(kFull, kept_dis));
    unsigned movers = __ballot_sync(kFull, moving);
    int cur = lane < k ? my_id : -1;
    float g = my_gate;
    while (movers) {   // warp-uniform
        const int r = __ffs(movers) - 1;
        movers &= movers - 1;
        const int fr = __shfl_sync(kFull, fin, r);
        const float gr = __shfl_sync(kFull, g, r);
        const unsigned holders = __ballot_sync(kFull, cur == fr);
        if (holders != 0u) {
            if (lane == __ffs(holders) - 1) g = __fadd_rn(g, gr);
            if (lane == r) {
                cur = -1;
                g = 0.f;
            }
            cnt4[1] += 1;
        } else {
            if (lane == r) cur = fr;
            cnt4[0] += 1;
        }
    }
    if (lane < k) {
        my_id = cur;
        my_gate = g;
    }
}

// Stage 3: SERE over the whole batch and the permutation.  The similarity
// copy into s_sim was issued by this CTA before it ranked its group.
template <int PL, bool SERE>
__device__ __forceinline__ void batch_tail(const RdArgs& a, float* s_sim, uint64_t* sim_bar, int* abort_flag,
                                           moe_dev_status* st) {
    constexpr int kWords = kRouteDispatchMaxT / 32;
    __shared__ uint32_t Pbits[kMaxPerLane], Ubefore[kMaxPerLane], Need[kMaxPerLane];
    __shared__ int Plist[MOE_MAX_EXPERTS], NeedList[MOE_MAX_EXPERTS];
    __shared__ int s_np, s_nn;
    __shared__ int wstat[kRdThreads / 32][4];
    __shared__ int tgt[MOE_MAX_EXPERTS];
    __shared__ uint32_t tkey[MOE_MAX_EXPERTS];
    __shared__ uint32_t bits[MOE_MAX_EXPERTS * kWords];
    __shared__ int cnt[MOE_MAX_EXPERTS];
    __shared__ int start[MOE_MAX_EXPERTS];
    __shared__ int s_id[kRouteDispatchMaxSlots];
    __shared__ float s_g[kRouteDispatchMaxSlots];
    __shared__ uint8_t s_prot[MOE_MAX_EXPERTS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = a.T, N = a.N, k = a.k;
    const int nw = (T + 31) / 32;
    const uint8_t* prot = (SERE && a.protect != nullptr) ? s_prot : nullptr;
    uint32_t* ws = reinterpret_cast<uint32_t*>(a.ws);
    if ((SERE || a.publish) && threadIdx.x < kMaxPerLane) {
        Pbits[threadIdx.x] = __ldcg(&ws[kWsP + threadIdx.x]);
        Ubefore[threadIdx.x] = __ldcg(&ws[kWsUb + threadIdx.x]);
        ws[kWsP + threadIdx.x] = 0u;    // consumed: zero for the next call
        ws[kWsUb + threadIdx.x] = 0u;
    }
    if (SERE && a.protect != nullptr && threadIdx.x < N) s_prot[threadIdx.x] = a.protect[threadIdx.x];
    for (int i = threadIdx.x; i < N * nw; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    if (a.publish && threadIdx.x == 0) {
        // the experts the decode FFN may start on now: SERE never takes a
        // primary away, so P is active whatever the reroute does; without
        // SERE the union of the ranked experts is the active set.  A SERE
        // union small enough for one wave of the FFN's phase-1 units is
        // published whole: SMs that would idle stream every candidate, and
        // an expert that then moves costs only its phase 1.  So is one within
        // two waves whose P would keep at most a third of a wave busy while
        // the experts outside P need more than a wave (they could not start
        // in a single wave after the final routing either).
        int nu = 0, np = 0;
        for (int w = 0; w < kMaxPerLane; ++w) {
            nu += __popc(Ubefore[w]);
            np += __popc(Pbits[w]);
        }
        const int sm = a.spec_max;
        const bool whole = !SERE || nu <= sm || (3 * np <= sm && nu - np > sm && nu <= 2 * sm);
        for (int w = 0; w < kMaxPerLane; ++w) ws[kWsEarly + 1 + w] = whole ? Ubefore[w] : Pbits[w];
        st_release_gpu(reinterpret_cast<int*>(ws) + kWsEarly, 1);
    }
    // bit t of expert e's presence bitmap marks token t holding e (a token
    // holds an expert at most once)
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const int id = __ldcg(&a.ids[i]);
        s_id[i] = id;
        s_g[i] = __ldcg(&a.gates[i]);
        if (!SERE && id >= 0 && id < N) atomicOr(&bits[id * nw + (i / k >> 5)], 1u << ((i / k) & 31));
    }
    __syncthreads();
    int cnt4[4] = {0, 0, 0, 0};
    if constexpr (SERE) {
        // the members of P, and the sources that need a target: experts held
        // as a slot, outside P, not protected
        if (warp == 0) {
            const int n = compact_bits(Pbits, N, Plist);
            if (lane == 0) s_np = n;
        } else if (warp == 1) {
            for (int w = 0; w < (N + 31) / 32; ++w) {
                const int e = 32 * w + lane;
                const bool need = e < N && (Ubefore[w] >> lane & 1u) && !(Pbits[w] >> lane & 1u) &&
                                  !(prot != nullptr && prot[e] != 0);
                const uint32_t b = __ballot_sync(kFull, need);
                if (lane == 0) Need[w] = b;
            }
            const int n = compact_bits(Need, N, NeedList);
            if (lane == 0) s_nn = n;
        }
        bool staged = a.stage_sim != 0;
        if (staged) {
            // every thread observes the copy's completion (bounded); on a
            // time-out the kernel records it and reads the similarity from
            // global memory
            if (!mbar_wait(smem_u32(sim_bar), 0, abort_flag, st, kSiteDrain)) staged = false;
        }
        staged = __syncthreads_and(staged ? 1 : 0) != 0;
        const float* simp = staged ? s_sim : a.sim;
        // each needed source's most similar member of P (ties to the lower
        // id: the list is ascending and the per-lane scan keeps the first)
        const int np = s_np, nn = s_nn;
        for (int i = warp; i < nn; i += kRdThreads / 32) {
            const int src = NeedList[i];
            const float* row = simp + static_cast<size_t>(src) * N;
            uint32_t bk = 0u;
            int bp = 0;
            for (int j = lane; j < np; j += 32) {
                const int p = Plist[j];
                const uint32_t key = order_key(row[p]);
                if (key > bk) {
                    bk = key;
                    bp = p;
                }
            }
            const uint32_t mk = __reduce_max_sync(kFull, bk);
            const uint32_t cand = (bk == mk && bk != 0u) ? static_cast<uint32_t>(bp) : 0xffffffffu;
            const int pbest = static_cast<int>(__reduce_min_sync(kFull, cand));
            if (lane == 0) {
                tgt[src] = pbest;
                tkey[src] = mk;
            }
        }
        __syncthreads();
        for (int t = warp; t < T; t += kRdThreads / 32) {
            int id = -1;
            float g = 0.f;
            if (lane < k) {
                id = s_id[t * k + lane];
                g = s_g[t * k + lane];
            }
            sere_token_movers(k, a.kp, a.rho, prot, Pbits, tgt, tkey, id, g, cnt4);
            if (lane < k) {
                s_id[t * k + lane] = id;
                s_g[t * k + lane] = g;
                a.ids[static_cast<size_t>(t) * k + lane] = id;
                a.gates[static_cast<size_t>(t) * k + lane] = g;
                if (id >= 0 && id < N) atomicOr(&bits[id * nw + (t >> 5)], 1u << (t & 31));
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) wstat[warp][i] = cnt4[i];
        }
        __syncthreads();
        if (threadIdx.x < (N + 31) / 32 && a.union_bitmap != nullptr) a.union_bitmap[threadIdx.x] = Pbits[threadIdx.x];
    }
    // the expert-sorted permutation of the final slots: a row's position is
    // start[e] plus the set bits below t in expert e's presence bitmap
    for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = block_count(bits, e, nw);
    __syncthreads();
    const int n_active = scan_experts_warps(cnt, N, a.counts, a.offsets, a.active, start);
    if (SERE && threadIdx.x == 0 && a.stats != nullptr) {
        int ub = 0, np = 0;
        for (int w = 0; w < kMaxPerLane; ++w) {
            ub += __popc(Ubefore[w]);
            np += __popc(Pbits[w]);
        }
        int sum4[4] = {0, 0, 0, 0};
        for (int w = 0; w < kRdThreads / 32; ++w)
            for (int i = 0; i < 4; ++i) sum4[i] += wstat[w][i];
        a.stats[0] = ub;
        a.stats[1] = np;
        a.stats[2] = n_active;   // the union after the reroute is the set of experts with rows
        for (int i = 0; i < 4; ++i) a.stats[3 + i] = sum4[i];
        a.stats[7] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const int e = s_id[i];
        if (e < 0) continue;
        if (e >= N) {
            report(st, MOE_DEV_BAD_INDEX, e);
            continue;
        }
        const int t = i / k, w0 = t >> 5;
        int c = __popc(bits[e * nw + w0] & ((1u << (t & 31)) - 1u));
        for (int w = 0; w < w0; ++w) c += __popc(bits[e * nw + w]);
        const int row = start[e] + c;
        a.row_token[row] = t;
        a.row_gate[row] = s_g[i];
    }
}

template <typename XT, int PL, bool SERE>
__global__ void __launch_bounds__(kRdThreads, 1) route_dispatch_kernel(const XT* __restrict__ x,
                                                                        const float* __restrict__ w, RdArgs a,
                                                                        moe_dev_status* st) {
    extern __shared__ __align__(16) float s_sim[];   // [N][N] when staged
    __shared__ float part[4 * kRdEpc][4];
    __shared__ bool s_last;
    __shared__ __align__(8) uint64_t sim_bar;
    __shared__ int abort_flag;
    // 1. this CTA's tile of router logits; its first W_r lines are requested
    // before the wait for the preceding launch (which does not write W_r)
    auto after_first_loads = [&]() {
        pdl_wait();
        if (a.publish && blockIdx.x == 0 && blockIdx.y == 0) {
            // the early flag goes back to zero before any CTA of this grid lets
            // the FFN launch, so the FFN can only see this call's publication
            if (threadIdx.x == 0) {
                a.ws[kWsEarly] = 0;
                __threadfence();
            }
            __syncthreads();
        }
        pdl_trigger();
        if (SERE && blockIdx.x == 0 && blockIdx.y == 0) {
            // pull the similarity into the L2 while the logits are computed
            const int lines = (a.N * a.N * 4 + 127) / 128;
            for (int l = threadIdx.x; l < lines; l += blockDim.x) prefetch_l2_keep(a.sim + l * 32);
        }
    };
    router_tile<XT, kRdEpc, (sizeof(XT) == 2 ? 4 : 2)>(x, w, a.T, a.H, a.N, blockIdx.x * kRdEpc, blockIdx.y * 4,
                                                         a.logits, part, after_first_loads);
    // the CTA's logit writes are published by its ticket (barrier, then an
    // acquire-release fetch-and-add by one thread)
    __syncthreads();
    int* gticket = a.ws + kWsGroups + blockIdx.y;
    if (threadIdx.x == 0) s_last = atom_add_acq_rel_gpu(gticket, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;   // uniform over the block
    // 2. the last CTA of this token group ranks the group's tokens; it starts
    // copying the similarity into its shared memory first, in case it also
    // turns out to be the last group
    const bool stage = SERE && a.stage_sim != 0;
    if (threadIdx.x == 0) {
        *gticket = 0;   // every CTA of the group has taken its ticket
        abort_flag = 0;
        if (stage) {
            const uint32_t bytes = static_cast<uint32_t>(a.N) * static_cast<uint32_t>(a.N) * 4u;
            mbar_init(smem_u32(&sim_bar), 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(smem_u32(&sim_bar), bytes);
            bulk_copy_g2s(smem_u32(s_sim), a.sim, bytes, smem_u32(&sim_bar));
        }
    }
    rank_group<PL, SERE>(a, blockIdx.y, st);
    __syncthreads();
    if (threadIdx.x == 0) s_last = atom_add_acq_rel_gpu(a.ws + kWsTicket, 1) == static_cast<int>(gridDim.y) - 1;
    __syncthreads();
    if (s_last) {
        // 3. the last group: SERE over the batch and the permutation
        batch_tail<PL, SERE>(a, s_sim, &sim_bar, &abort_flag, st);
    }
    // the copy lands before this CTA's shared memory is released (bounded)
    if (stage && threadIdx.x == 0) mbar_drain(smem_u32(&sim_bar), 0);
    if (!s_last) return;
    if (threadIdx.x == 0) a.ws[kWsTicket] = 0;   // every group has taken its ticket
}

template <typename XT, int PL>
static cudaError_t rd_launch(const XT* x, const float* w, const RdArgs& a, bool sere, moe_dev_status* st,
                             cudaStream_t s) {
    const dim3 grid((a.N + kRdEpc - 1) / kRdEpc, (a.T + 3) / 4);
    const size_t smem = a.stage_sim ? static_cast<size_t>(a.N) * a.N * 4 : 0;
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int dev = 0;
    cudaGetDevice(&dev);
    if (sere && dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(route_dispatch_kernel<XT, PL, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kRdStageN * kRdStageN * 4);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    if (sere) return launch_pdl(route_dispatch_kernel<XT, PL, true>, grid, dim3(kRdThreads), smem, s, x, w, a, st);
    return launch_pdl(route_dispatch_kernel<XT, PL, false>, grid, dim3(kRdThreads), 0, s, x, w, a, st);
}

template <typename XT>
static cudaError_t rd_launch_pl(const XT* x, const float* w, const RdArgs& a, bool sere, moe_dev_status* st,
                                cudaStream_t s) {
    if (a.N <= 32) return rd_launch<XT, 1>(x, w, a, sere, st, s);
    if (a.N <= 64) return rd_launch<XT, 2>(x, w, a, sere, st, s);
    if (a.N <= 128) return rd_launch<XT, 4>(x, w, a, sere, st, s);
    return rd_launch<XT, 8>(x, w, a, sere, st, s);
}

cudaError_t launch_route_dispatch(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int k,
                                  bool renorm, float* logits, int32_t* ids, float* gates, const moe_sere_params* sere,
                                  int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_gate,
                                  int32_t* active, void* ws, bool publish_early, moe_dev_status* st,
                                  cudaStream_t s, int spec_union_max) {
    RdArgs a{};
    a.publish = publish_early ? 1 : 0;
    a.spec_max = spec_union_max;
    a.T = T;
    a.H = H;
    a.N = N;
    a.k = k;
    a.renorm = renorm ? 1 : 0;
    if (sere != nullptr) {
        a.kp = sere->k_primary;
        a.rho = sere->rho;
        a.sim = sere->sim;
        a.protect = sere->protect;
        a.union_bitmap = sere->union_bitmap;
        a.stats = sere->stats;
        a.stage_sim = (N <= kRdStageN && (reinterpret_cast<uintptr_t>(sere->sim) & 15u) == 0) ? 1 : 0;
    }
    a.logits = logits;
    a.ids = ids;
    a.gates = gates;
    a.counts = counts;
    a.offsets = offsets;
    a.row_token = row_token;
    a.row_gate = row_gate;
    a.active = active;
    a.ws = static_cast<int*>(ws);
    if (x_dtype == MOE_DTYPE_BF16)
        return rd_launch_pl(static_cast<const __nv_bfloat16*>(x), w_router, a, sere != nullptr, st, s);
    return rd_launch_pl(static_cast<const float*>(x), w_router, a, sere != nullptr, st, s);
}

}  // namespace moe
