// ffn_decode.cu -- the decode FFN: the grouped SwiGLU expert FFN with the
// weighted combine fused in, for batches of up to 64 tokens.
//
// E_j(x) = W_down_j (silu(W_gate_j x) * (W_up_j x)) and
// y(x) = sum_j G(x)_j E_j(x): "MACS: Modality-Aware Capacity Scaling for
// Efficient Multimodal MoE Inference", sec. 3.1, Eq. (1).  Decode moves every
// active expert's weights once and little else (the SERE article, sec. 1.2 and
// 2.2), so the kernel is built to keep HBM streaming from its first
// microsecond to its last:
//
//  * All-token units.  A unit multiplies one weight tile by the whole batch:
//    the token operand of every stage is one TMA box of x (NT rows, rows past
//    the batch read as zero), never a gather of the expert's rows.  Four-row
//    gathers cost a stage more time in the TMA unit than its 32 KiB of
//    weights, which capped one SM's stream at ~48 GB/s; boxes let an SM pull
//    well over 70 GB/s when others are idle.  Only the routed tokens' columns
//    of the result are used.
//  * Expert-indexed activations.  Phase 1 of expert e writes A[e*NT + t][:]
//    and counts its units in done[e]; nothing in phase 1 depends on the
//    routing beyond the expert id.
//  * Early start.  When the routing launch publishes its early experts (the
//    primary union P of SERE, the whole union before the reroute when its
//    phase-1 units fit one wave, or the union for plain top-k) as soon as
//    ranking ends, the kernel streams those experts' phase 1 while the
//    routing launch still reroutes and permutes; only the remaining experts'
//    phase 1 and the down projections wait for the final routing, which a
//    scheduler warp reads (griddepcontrol.wait) and tabulates.
//
// Units, handed out by a global counter after a static first unit per CTA:
//   [0, nE*S)          phase 1 of the early experts (S units each),
//   [nE*S, n1)         phase 1 of the other active experts,
//   [n1, n1 + nA*MT*KP)  phase 2: per active expert, per 128-row H-tile of
//                      W_down (and per K half when small batches leave SMs
//                      idle): gate * W_down A^T added into y.
// A phase-1 unit is a half slice: 64 gate rows and the same 64 up rows of
// W_gate and W_up, stacked as one 128-row MMA operand, over K = H (S = I/64
// units per expert); the epilogue pairs each gate row with its up row
// through shared memory.  A phase-2 unit waits (bounded, acquire) until its
// expert's S phase-1 units have published A.  The warp roles are those of
// the weight-major kernel in ffn.cu.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace moe {

namespace {

__device__ __forceinline__ float silu_mul_d(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <int NT>
struct DcCfg {
    static constexpr int BH = 128;                  // H-tile of a phase-2 unit (MMA M)
    static constexpr int BK = 64;                   // one 128-byte swizzle row of bf16
    static constexpr int W_BOX = 128 * 64 * 2;      // 16 KiB
    static constexpr int W_BYTES = 2 * W_BOX;       // weights per stage
    static constexpr int X_ATOM = NT * 128;         // NT token rows of one 64-column K chunk
    static constexpr int X_BYTES = 2 * X_ATOM;      // every stage takes two K chunks
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int NSTAGE = NT <= 32 ? 5 : 4;
    static constexpr int EPI_WARPS = 8;             // two warps per TMEM lane quadrant
    static constexpr int SCHED_WARP = 2 + EPI_WARPS;
    static constexpr int THREADS = 32 * (SCHED_WARP + 1);
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int CW = NT / 2;               // token columns per epilogue warp
    static constexpr int QN = 4;                    // unit ids in flight between the warp roles
    static constexpr int NBAR = 2 * NSTAGE + 6 + 2 * QN;
    static constexpr int MISC_INTS = 16;
    static constexpr int RT_CAP = NT * MOE_MAX_RANKS;   // every dispatch row (T <= NT, k <= 16)
    static constexpr int LIST_INTS = 3 * MOE_MAX_EXPERTS + (MOE_MAX_EXPERTS + 1) + 2 * (MOE_MAX_EXPERTS / 32);
    static constexpr int XCH_BYTES = 64 * NT * 4;  // the up rows of a phase-1 unit, [NT][64] fp32
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + NBAR * 8 + MISC_INTS * 4 + LIST_INTS * 4 +
                                EPI_WARPS * 32 * 8 + XCH_BYTES + RT_CAP * 8;
    static constexpr uint32_t TMEM_COLS = 2 * NT;   // two accumulator slots of NT columns
    static_assert(STAGE % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128, "TMEM allocation");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(CW == 8 || CW == 16 || CW == 32, "epilogue column split");
};

// Compacts the set bits e < N of bm[0 .. ceil(N/32)) into list (ascending)
// with one warp; returns the count.
__device__ __forceinline__ int compact_experts(const uint32_t* bm, int N, int* list) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    for (int w = 0; w < (N + 31) / 32; ++w) {
        uint32_t b = bm[w];
        if (32 * w + 32 > N) b &= (1u << (N - 32 * w)) - 1u;
        if (b >> lane & 1u) list[base + __popc(b & ((1u << lane) - 1u))] = 32 * w + lane;
        base += __popc(b);
    }
    return base;
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(DcCfg<NT>::THREADS, 1)
    ffn_decode_kernel(const __grid_constant__ CUtensorMap tm_wg64, const __grid_constant__ CUtensorMap tm_wu64,
                      const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_act, const int32_t* __restrict__ offsets,
                      const int32_t* __restrict__ active, const int32_t* __restrict__ row_token,
                      const float* __restrict__ row_gate, const uint32_t* early, __nv_bfloat16* __restrict__ act_g,
                      int* counters, float* __restrict__ out, float* __restrict__ y_zero, int T, int H, int I, int N,
                      int k, int fuse_combine, moe_dev_status* st) {
    using C = DcCfg<NT>;
    constexpr int CW = C::CW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::NSTAGE * C::STAGE);
    int* misc = reinterpret_cast<int*>(bars + C::NBAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = misc + 1;
    volatile int* uring = misc + 2;                  // [QN] unit ids, -1 = no more work
    int* s_cnt = misc + 2 + C::QN;                   // nE, nL, nA, n1, n_total, KP2, last-CTA flag
    int* elist = misc + C::MISC_INTS;                // [N] early experts, ascending
    int* llist = elist + MOE_MAX_EXPERTS;            // [N] other active experts, ascending
    int* alist = llist + MOE_MAX_EXPERTS;            // [N] active experts, in phase-2 order
    int* s_off = alist + MOE_MAX_EXPERTS;            // [N + 1] dispatch offsets
    uint32_t* ebits = reinterpret_cast<uint32_t*>(s_off + MOE_MAX_EXPERTS + 1);   // early bitmap
    uint32_t* abits = ebits + MOE_MAX_EXPERTS / 32;                                // active bitmap
    int* etok_all = reinterpret_cast<int*>(abits + MOE_MAX_EXPERTS / 32);         // [EPI_WARPS][32]
    float* egt_all = reinterpret_cast<float*>(etok_all + C::EPI_WARPS * 32);      // [EPI_WARPS][32]
    float* xch = egt_all + C::EPI_WARPS * 32;                                      // [NT][64] half units
    int* s_rt = reinterpret_cast<int*>(xch + C::XCH_BYTES / 4);                    // [RT_CAP] row -> token
    float* s_rg = reinterpret_cast<float*>(s_rt + C::RT_CAP);                      // [RT_CAP] row -> gate

    const uint32_t ring_a = smem_u32(ring);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_ACCF = 2 * C::NSTAGE, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2,
              B_TABLE = B_DRAIN + 1, B_QFULL = B_TABLE + 1, B_QEMPTY = B_QFULL + C::QN;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_ACCF + b), 1);
            mbar_init(bar(B_ACCE + b), C::EPI_THREADS);
        }
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_TABLE), 1);
        for (int i = 0; i < C::QN; ++i) {
            mbar_init(bar(B_QFULL + i), 1);
            mbar_init(bar(B_QEMPTY + i), 2);   // the MMA thread and the epilogue
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_wg64);
        tma_prefetch_desc(&tm_wu64);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_act);
    }
    // Without an early list everything waits for the preceding launch here.
    // With one, the preceding launch is the routing launch, which has already
    // waited for everything before it (so x is final), never waits for this
    // kernel, and is fully resident before this kernel starts; only its
    // final outputs are read after griddepcontrol.wait (scheduler warp).
    if (early == nullptr) pdl_wait();
    pdl_trigger();
    const int nw = (N + 31) / 32;
    if (warp == 0) {
        // the experts phase 1 may start on at once: the routing launch's
        // early list, or without one the dispatch's whole active list (one
        // round trip of independent loads)
        if (lane < nw) ebits[lane] = 0u;
        __syncwarp();
        if (early != nullptr) {
            int have = 0;
            if (lane == 0) {
                const unsigned long long t0 = global_ns();
                while (true) {
                    if (ld_acquire_gpu(reinterpret_cast<const int*>(early)) != 0) {
                        have = 1;
                        break;
                    }
                    if (global_ns() - t0 > kWaitLimitNs) {
                        report(st, MOE_DEV_TIMEOUT, kSiteDependency);
                        break;
                    }
                    __nanosleep(32);
                }
            }
            have = __shfl_sync(kFull, have, 0);
            if (have && lane < nw) ebits[lane] = __ldcg(early + 1 + lane);
        } else {
            int cnt = 0;
            for (int i = lane; i <= N; i += 32) {
                const int v = active[i];
                if (i == 0) cnt = v;
                else llist[i - 1] = (v >= 0 && v < N) ? v : -1;
            }
            cnt = __shfl_sync(kFull, cnt, 0);
            cnt = cnt < 0 ? 0 : (cnt > N ? N : cnt);
            __syncwarp();
            for (int a = lane; a < cnt; a += 32) {
                const int e = llist[a];
                if (e >= 0) atomicOr(&ebits[e >> 5], 1u << (e & 31));
            }
        }
        __syncwarp();
        const int n = compact_experts(ebits, N, elist);
        if (lane == 0) s_cnt[0] = n;
    }
    __syncthreads();
    const int nE = s_cnt[0];
    const int S = I / 64;                      // phase-1 units (half slices) per expert
    const int MT = H / C::BH;
    const int KT1 = H / C::BK;
    const int KT2 = I / (2 * C::BK);
    const int nEU = nE * S;                    // early units
    const int ncol = min(NT, max(16, (T + 15) & ~15));   // MMA N: the batch rounded up to 16
    const int M = T * k;
    int* const work_head = counters;
    int* const done = counters + 1;            // [N] phase-1 units finished per expert
    int* const zero_claim = counters + 1 + N;  // 4 KiB chunks of y handed out for zeroing
    int* const zero_done = zero_claim + 1;     // chunks of y zeroed
    int* const exit_cnt = zero_done + 1;       // CTAs that have finished
    constexpr int kZeroChunk = 1024;           // floats per chunk of y
    const long long y_elems = static_cast<long long>(T) * H;
    const int n_zchunks = (y_zero != nullptr) ? static_cast<int>((y_elems + kZeroChunk - 1) / kZeroChunk) : 0;

    // The final table, read once it is built: n1 (phase-1 units), n_total, KP2.
    struct Unit {
        bool p1;
        int e, sub, part;      // expert, I-slice or H-tile, K part of a phase-2 unit
        int row0, cnt;         // phase 2: the expert's dispatch rows
    };
    auto decode = [&](int u, Unit& d) {
        if (u < nEU) {
            d.p1 = true;
            d.e = elist[u / S];
            d.sub = u % S;
            d.part = 0;
            return;
        }
        const int n1 = s_cnt[3];
        if (u < n1) {
            const int v = u - nEU;
            d.p1 = true;
            d.e = llist[v / S];
            d.sub = v % S;
            d.part = 0;
            return;
        }
        const int kp = s_cnt[5];
        const int v = u - n1;
        const int a = v / (MT * kp);
        const int r = v - a * MT * kp;
        d.p1 = false;
        d.e = alist[a];
        d.sub = r / kp;
        d.part = r - d.sub * kp;
        d.row0 = s_off[d.e];
        d.cnt = s_off[d.e + 1] - d.row0;
    };
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The final routing, staged in shared memory by the epilogue and
    // scheduler warps together (their loads all in flight at once): active[]
    // (count, then ids, in llist for now), offsets[] and every dispatch row's
    // token and gate.  The epilogue warps arrive here after zeroing y; in
    // early mode they have nothing else to do until the first accumulator.
    auto stage_routing = [&]() {
        constexpr int kStagers = 32 * (C::EPI_WARPS + 1);
        const int tid = threadIdx.x - 64;
        pdl_wait();
        for (int i = tid; i <= N; i += kStagers) {
            const int av = active[i];
            const int ov = offsets[i];
            s_off[i] = ov;
            if (i == 0) s_cnt[2] = av;
            else llist[i - 1] = av;
        }
        const int mrows = M <= C::RT_CAP ? M : C::RT_CAP;
        for (int i = tid; i < mrows; i += kStagers) {
            const int rt = row_token[i];
            const float rg = row_gate[i];
            s_rt[i] = rt;
            s_rg[i] = rg;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(kStagers) : "memory");
    };

    if (warp == C::SCHED_WARP) {
        // ---------------- scheduler: the final routing -> table ----------------
        stage_routing();
        int na = s_cnt[2];
        bool bad = na < 0 || na > N || M > C::RT_CAP;
        if (bad) na = 0;
        // the dispatch's active list: ids in range, rows within [0, T k), each
        // expert holding each token at most once (at most T rows)
        for (int a = lane; a < na; a += 32) {
            const int e = llist[a];
            if (e < 0 || e >= N) {
                bad = true;
                continue;
            }
            const int r0 = s_off[e], c = s_off[e + 1] - r0;
            if (r0 < 0 || c <= 0 || c > T || r0 + c > M) bad = true;
        }
        bad = __any_sync(kFull, bad);
        __syncwarp();
        if (bad) na = 0;
        for (int a = lane; a < na; a += 32) alist[a] = llist[a];
        __syncwarp();
        // the active experts outside the early list, ascending
        int nl = 0;
        for (int base = 0; base < na; base += 32) {
            const int a = base + lane;
            const int e = a < na ? alist[a] : 0;
            const bool late = a < na && !(ebits[e >> 5] >> (e & 31) & 1u);
            const unsigned m = __ballot_sync(kFull, late);
            if (late) llist[nl + __popc(m & ((1u << lane) - 1u))] = e;
            nl += __popc(m);
        }
        // Phase 2 visits the experts in the order their phase 1 was handed out:
        // the early experts that are active, then the others.  A down
        // projection handed out right after the first wave of phase-1 units
        // then belongs to an expert whose activations are (nearly) published,
        // instead of waiting for an expert whose phase 1 runs in the last wave.
        if (lane < nw) abits[lane] = 0u;
        __syncwarp();
        for (int a = lane; a < na; a += 32) atomicOr(&abits[alist[a] >> 5], 1u << (alist[a] & 31));
        __syncwarp();
        int np = 0;
        for (int base = 0; base < nE; base += 32) {
            const int a = base + lane;
            const int e = a < nE ? elist[a] : 0;
            const bool act = a < nE && (abits[e >> 5] >> (e & 31) & 1u);
            const unsigned m = __ballot_sync(kFull, act);
            if (act) alist[np + __popc(m & ((1u << lane) - 1u))] = e;
            np += __popc(m);
        }
        for (int a = lane; a < nl; a += 32) alist[np + a] = llist[a];
        __syncwarp();
        if (lane == 0) {
            if (bad) report(st, MOE_DEV_BAD_INDEX, s_cnt[2]);
            const int n1 = (nE + nl) * S;
            // phase-2 K halves when whole tiles would leave SMs idle (small batches)
            const int kp = (KT2 % 2 == 0 && na * MT < 2 * static_cast<int>(gridDim.x)) ? 2 : 1;
            s_cnt[1] = nl;
            s_cnt[2] = na;
            s_cnt[3] = n1;
            s_cnt[4] = n1 + na * MT * kp;
            s_cnt[5] = kp;
            mbar_arrive(bar(B_TABLE));
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------- TMA producer (lane 0 issues) ----------------
        const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, pend = 0, pend_par = 0;
        bool ok = true, table = false;
        int cur = blockIdx.x;   // static first unit; later ones from the work counter
        for (int j = 0;; ++j) {
            int n_total = 0;
            if (lane == 0) {
                if (cur >= nEU && !table) {
                    ok = mbar_wait(bar(B_TABLE), 0, abort_flag, st, kSiteDependency);
                    table = ok;
                }
                n_total = table ? s_cnt[4] : nEU;
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            n_total = __shfl_sync(kFull, n_total, 0);
            const bool fin = cur >= n_total;
            if (lane == 0) {
                // hand the unit (or the end mark) to the MMA and epilogue warps
                const int qs = j % C::QN;
                ok = mbar_wait(bar(B_QEMPTY + qs), ((j / C::QN) & 1) ^ 1, abort_flag, st, kSiteProducerEmpty);
                if (ok) {
                    uring[qs] = fin ? -1 : cur;
                    mbar_arrive(bar(B_QFULL + qs));
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok || fin) break;
            int nxt = 0;
            if (lane == 0) {
                Unit d;
                decode(cur, d);
                if (!d.p1) {
                    // A of this expert: all S phase-1 units must have published it
                    const unsigned long long t0 = global_ns();
                    while (ld_acquire_gpu(done + d.e) < S ||
                           (n_zchunks > 0 && ld_acquire_gpu(zero_done) < n_zchunks)) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (global_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            report(st, MOE_DEV_TIMEOUT, kSiteDependency);
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    fence_proxy_async_global();
                }
                const int nk = d.p1 ? KT1 / 2 : KT2 / s_cnt[5];
                // the next unit is reserved two stages before this one's last: late
                // enough that a CTA near the end of the queue holds as little work
                // that an idle SM could have taken, early enough to hide the
                // counter's round trip (a loop that stops early reserves nothing,
                // and the CTA then stops too)
                const int kres = nk > 2 ? nk - 2 : 0;
                for (int kt = 0; kt < nk && ok; ++kt) {
                    if (kt == kres) nxt = atomicAdd(work_head, 1) + static_cast<int>(gridDim.x);
                    if (!mbar_wait(bar(B_EMPTY + stage), phase ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring_a + stage * C::STAGE;
                    const uint32_t fb = bar(B_FULL + stage);
                    if (d.p1) {
                        // two 64-column K chunks; each is [64 gate rows; the same 64 up rows]
                        const int wrow = d.e * I + d.sub * 64;
                        mbar_arrive_expect_tx(fb, C::W_BYTES + 2 * C::X_ATOM);
                        for (int c = 0; c < 2; ++c) {
                            const int kc = kt * 2 * C::BK + c * C::BK;
                            tma_load_2d(dst + c * C::W_BOX, &tm_wg64, kc, wrow, fb, pol_w);
                            tma_load_2d(dst + c * C::W_BOX + C::W_BOX / 2, &tm_wu64, kc, wrow, fb, pol_w);
                            tma_load_2d(dst + C::W_BYTES + c * C::X_ATOM, &tm_x, kc, 0, fb, pol_x);
                        }
                    } else {
                        const int wrow = d.e * H + d.sub * C::BH;
                        const int kc = (d.part * nk + kt) * 2 * C::BK;   // first K column of this stage
                        mbar_arrive_expect_tx(fb, C::W_BYTES + 2 * C::X_ATOM);
                        tma_load_2d(dst, &tm_wd, kc, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wd, kc + C::BK, wrow, fb, pol_w);
                        // the expert's activations for the whole batch: rows e * NT ..
                        for (int a = 0; a < 2; ++a)
                            tma_load_2d(dst + C::W_BYTES + a * C::X_ATOM, &tm_act, kc + a * C::BK, d.e * NT, fb,
                                        pol_x);
                    }
                    pend |= 1u << stage;
                    pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            cur = __shfl_sync(kFull, nxt, 0);
        }
        if (!ok && lane == 0) {
            // let every copy still in flight land before the CTA exits
            for (int i = 0; i < C::NSTAGE; ++i)
                if (pend >> i & 1u) mbar_drain(bar(B_FULL + i), pend_par >> i & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, table = false;
            const uint32_t idesc = idesc_bf16_f32(128, ncol);
            for (int j = 0; ok; ++j) {
                const int qs = j % C::QN;
                if (!mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteMmaFull)) break;
                const int un = uring[qs];
                mbar_arrive(bar(B_QEMPTY + qs));
                if (un < 0) break;
                if (un >= nEU && !table) {
                    if (!mbar_wait(bar(B_TABLE), 0, abort_flag, st, kSiteMmaFull)) break;
                    table = true;
                }
                const bool p1 = un < (table ? s_cnt[3] : nEU);
                const int b = j & 1;
                const uint32_t acc0 = tmem + b * NT;
                if (!mbar_wait(bar(B_ACCE + b), ((j >> 1) & 1) ^ 1, abort_flag, st, kSiteMmaTmemFree)) break;
                tc_fence_after();
                const int nk = p1 ? KT1 / 2 : KT2 / s_cnt[5];
                for (int kt = 0; kt < nk; ++kt) {
                    if (!mbar_wait(bar(B_FULL + stage), phase, abort_flag, st, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring_a + stage * C::STAGE;
                    // two K chunks: 128 weight rows (phase 1: 64 gate and 64 up rows
                    // stacked) against the NT token columns of the same chunk
#pragma unroll
                    for (int kk = 0; kk < 2 * C::BK / 16; ++kk) {
                        const uint64_t dw = sw128_desc(a + (kk >> 2) * C::W_BOX + (kk & 3) * 32);
                        const uint64_t dx = sw128_desc(a + C::W_BYTES + (kk >> 2) * C::X_ATOM + (kk & 3) * 32);
                        tc_mma_bf16(acc0, dw, dx, idesc, (kt | kk) != 0);
                    }
                    tc_commit(bar(B_EMPTY + stage));
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar(B_ACCF + b));
            }
            // every issued MMA has finished before TMEM is released
            tc_commit(bar(B_DRAIN));
            mbar_drain(bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..9, two per TMEM lane quadrant ----------------
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;              // which half of the token columns
        const int row = q * 32 + lane;                 // row of the 128-row tile (I row or H row)
        const int c_lo = half * CW;                    // first token column of this warp
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        int* etok = etok_all + (warp - 2) * 32;
        float* egt = egt_all + (warp - 2) * 32;
        bool table = false;
        // zero y (MOE_FFN_ZERO_Y) in chunks that running warps claim, before
        // the first accumulator is ready; phase-2 units wait for all chunks
        while (n_zchunks > 0) {   // warp-uniform
            int c = (lane == 0) ? atomicAdd(zero_claim, 1) : 0;
            c = __shfl_sync(kFull, c, 0);
            if (c >= n_zchunks) break;
            const long long beg = static_cast<long long>(c) * kZeroChunk;
            const long long end = min(beg + kZeroChunk, y_elems);
            for (long long i = beg + lane * 4; i < end; i += 128)
                *reinterpret_cast<float4*>(y_zero + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            __syncwarp();
            if (lane == 0) red_release_gpu_add(zero_done, 1);
        }
        stage_routing();
        for (int j = 0;; ++j) {
            const int qs = j % C::QN;
            // every lane polls; the warp proceeds only if all lanes saw the phase complete
            bool okw = __all_sync(kFull, mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteEpiG1Done));
            const int un = okw ? uring[qs] : -1;
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (un < 0) break;   // the same value in every epilogue thread
            if (un >= nEU && !table) {
                okw = __all_sync(kFull, mbar_wait(bar(B_TABLE), 0, abort_flag, st, kSiteEpiG1Done));
                table = okw;
            }
            Unit d{};
            if (okw) decode(un, d);
            const int b = j & 1;
            const uint32_t acc0 = tmem + b * NT;
            okw = __all_sync(kFull, okw && mbar_wait(bar(B_ACCF + b), (j >> 1) & 1, abort_flag, st, kSiteEpiG1Done));
            if (d.p1) {
                // accumulator lanes 0-63: gate rows, 64-127: the same up rows.  The
                // up warps stage their values in shared memory; after a barrier of
                // all epilogue warps (taken by every warp) the gate warps form the
                // SwiGLU for the 64 I rows of the unit.
                if (okw && q >= 2) {
                    tc_fence_after();
#pragma unroll
                    for (int c8 = 0; c8 < CW / 8; ++c8) {
                        if (c_lo + c8 * 8 >= ncol) break;   // warp-uniform
                        uint32_t u[8];
                        tmem_ld8(acc0 + lane_off + c_lo + c8 * 8, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            xch[(c_lo + c8 * 8 + jj) * 64 + (q - 2) * 32 + lane] = __uint_as_float(u[jj]);
                    }
                    tc_fence_before();
                    mbar_arrive(bar(B_ACCE + b));
                }
                okw = named_sync_and(C::EPI_THREADS, okw);
                if (okw && q < 2) {
                    tc_fence_after();
                    __nv_bfloat16* dst = act_g + static_cast<size_t>(d.e) * NT * I + d.sub * 64 + row;
#pragma unroll
                    for (int c8 = 0; c8 < CW / 8; ++c8) {
                        if (c_lo + c8 * 8 >= ncol) break;   // warp-uniform
                        uint32_t g[8];
                        tmem_ld8(acc0 + lane_off + c_lo + c8 * 8, g);
                        tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int t = c_lo + c8 * 8 + jj;
                            dst[static_cast<size_t>(t) * I] =
                                __float2bfloat16_rn(silu_mul_d(__uint_as_float(g[jj]), xch[t * 64 + row]));
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(bar(B_ACCE + b));
                    fence_proxy_async_global();
                    __threadfence();
                }
            } else if (okw) {
                tc_fence_after();
                // column c_lo + js is token c_lo + js: etok[js] = its dispatch row
                // for this expert, or -1 when the token was not routed here
                if (lane < CW) etok[lane] = -1;
                __syncwarp();
                for (int jr = lane; jr < d.cnt; jr += 32) {
                    const int r = d.row0 + jr;
                    const int t = s_rt[r];
                    if (t >= c_lo && t < c_lo + CW && t < T) {
                        etok[t - c_lo] = r;
                        egt[t - c_lo] = s_rg[r];
                    }
                }
                __syncwarp();
                // read the accumulator in chunks of up to 16 columns; it is released right
                // after the last read, before the last chunk's reductions
                constexpr int CH = CW < 16 ? CW : 16;
                const int h = d.sub * C::BH + row;
#pragma unroll
                for (int c16 = 0; c16 < CW / CH; ++c16) {
                    const bool any = c_lo + c16 * CH < ncol;   // warp-uniform
                    uint32_t vv[CH];
                    if (any) {
                        if constexpr (CH == 8) {
                            tmem_ld8(acc0 + lane_off + c_lo, vv);
                        } else {
                            tmem_ld16(acc0 + lane_off + c_lo + c16 * CH, vv);
                        }
                        tmem_ld_wait();
                    }
                    if (c16 == CW / CH - 1) {
                        tc_fence_before();
                        mbar_arrive(bar(B_ACCE + b));
                    }
                    if (!any) continue;
#pragma unroll
                    for (int jj = 0; jj < CH; ++jj) {
                        const int js = c16 * CH + jj;
                        const int r = etok[js];
                        if (r >= 0) {
                            if (fuse_combine)
                                atomicAdd(out + static_cast<size_t>(c_lo + js) * H + h,
                                          egt[js] * __uint_as_float(vv[jj]));
                            else
                                atomicAdd(out + static_cast<size_t>(r) * H + h, __uint_as_float(vv[jj]));
                        }
                    }
                }
            }
            // all epilogue warps pass here once per unit; a failure anywhere ends them together
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (threadIdx.x == 64) {
                if (d.p1) red_release_gpu_add(done + d.e, 1);
                mbar_arrive(bar(B_QEMPTY + qs));   // every epilogue thread has read the unit id
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // the last CTA to finish returns the counters to zero for the next call
    __syncthreads();
    if (threadIdx.x == 0) s_cnt[6] = atom_add_acq_rel_gpu(exit_cnt, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (s_cnt[6])
        for (int i = threadIdx.x; i < N + 4; i += blockDim.x) counters[i] = 0;
}

// Rows of the decode kernel's activation buffer: NT per expert.
long long ffn_decode_act_rows(int T, int N) { return static_cast<long long>(N) * ffn_decode_nt(T); }

template <int NT>
static cudaError_t run_decode(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                              int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                              const int32_t* active, const uint32_t* early, uint32_t flags, float* out, void* ws,
                              moe_dev_status* st, cudaStream_t s) {
    using C = DcCfg<NT>;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    int* counters = static_cast<int*>(ws);
    __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + ffn_decode_ctr_bytes());
    float* y_zero = (fuse && (flags & MOE_FFN_ZERO_Y)) ? out : nullptr;
    CUtensorMap tm_wg64, tm_wu64, tm_wd, tm_x, tm_act;
    if (!make_tmap(&tm_wg64, wg, H, static_cast<uint64_t>(N) * I, 64, 64) ||
        !make_tmap(&tm_wu64, wu, H, static_cast<uint64_t>(N) * I, 64, 64) ||
        !make_tmap(&tm_wd, wd, I, static_cast<uint64_t>(N) * H, 64, 128) ||
        // the whole batch as one box of NT rows (rows past T read as zero)
        !make_tmap(&tm_x, x, H, static_cast<uint64_t>(T), 64, NT) ||
        !make_tmap(&tm_act, act, I, static_cast<uint64_t>(ffn_decode_act_rows(T, N)), 64, NT))
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int devi = 0;
    cudaError_t e = cudaGetDevice(&devi);
    if (e != cudaSuccess) return e;
    if (devi < 0 || devi >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[devi]) {
        e = cudaFuncSetAttribute(ffn_decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[devi] = true;
    }
    return launch_pdl(ffn_decode_kernel<NT>, dim3(sm_count()), dim3(C::THREADS), C::SMEM, s, tm_wg64, tm_wu64,
                      tm_wd, tm_x, tm_act, offsets, active, row_token, row_gate, early, act,
                      counters, out, y_zero, T, H, I, N, k, fuse ? 1 : 0, st);
}

// Phase-1 units are half slices (64 gate and 64 up rows) at every batch: a
// few dozen active experts give only a wave or two of whole 128-row
// I-slices (fewer than the SMs when T*k or N is small), so the experts whose
// phase 1 falls in the last, partial wave would hold up their down
// projections; twice the units let the work counter even out SMs that
// stream at different rates.
int ffn_decode_units_per_expert(int T, int I, int N, int k) {
    (void)T;
    (void)N;
    (void)k;
    return I / 64;
}

int ffn_decode_one_wave_experts(int T, int I, int N, int k) {
    return sm_count() / ffn_decode_units_per_expert(T, I, N, k);
}

cudaError_t launch_ffn_decode(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                              int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                              const int32_t* active, const uint32_t* early, uint32_t flags, float* out, void* ws,
                              moe_dev_status* st, cudaStream_t s) {
    if (T < 1 || T > kDecodeMaxT || k > MOE_MAX_RANKS || N > MOE_MAX_EXPERTS) return cudaErrorInvalidValue;
    switch (ffn_decode_nt(T)) {
        case 16:
            return run_decode<16>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, early, flags,
                                  out, ws, st, s);
        case 32:
            return run_decode<32>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, early, flags,
                                  out, ws, st, s);
        default:
            return run_decode<64>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, early, flags,
                                  out, ws, st, s);
    }
}

}  // namespace moe
