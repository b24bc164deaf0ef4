// ffn.cu -- grouped SwiGLU expert FFN with the weighted combine fused in.
//
// E_j(x) = W_down_j (silu(W_gate_j x) * (W_up_j x)) and
// y(x) = sum_j G(x)_j E_j(x): "MACS: Modality-Aware Capacity Scaling for
// Efficient Multimodal MoE Inference", sec. 3.1, Eq. (1).  Only the experts
// that received rows are visited, so the bytes moved per layer are the
// active experts' weights (the decode bottleneck the SERE article measures in
// sec. 1.2 / 2.2).
//
// bf16 path (tensor cores), by batch size:
//  * up to 64 tokens with k <= 16: the decode kernel of ffn_decode.cu;
//  * otherwise up to 1023 tokens: ffn_stream_kernel below, one persistent CTA per SM
//    with the weights as the 128-row MMA operand and each expert's rows, in
//    chunks of 64 gathered per stage, as the N operand;
//  * 1024 tokens and more: the token-major kernels (prefill).
// fp32 path: a CUDA-core kernel, one CTA per row.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace moe {


// Batches of at least this many tokens run the token-major kernels (about 64
// rows per expert at top-8 of 128); smaller ones the weight-major one.
constexpr int kTokenMajorMinT = 1024;
constexpr int kTmRows = 128;   // token rows per item of the token-major kernel (its MMA M)
constexpr int kTmCols = 256;   // its MMA N (H-tile of the down projection)

static bool token_major(int T, int H) { return T >= kTokenMajorMinT && H % kTmCols == 0; }

// Token-chunk width of the weight-major kernel.
constexpr int kStreamNT = 64;

// Upper bound on the items (expert, chunk of <= nt rows) of a dispatch of M rows.
static long long ffn_max_items(int T, int N, int k, int nt) {
    const long long M = static_cast<long long>(T) * k;
    return (N < M ? N : M) + (M + nt - 1) / nt;
}

static size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// The weight-major kernel's counters sit at the start of every bf16 FFN
// workspace, in a region of fixed size that nothing else writes, so that a
// workspace stays valid across calls of any batch size and either path.
// Items of the weight-major path: min(N, T k) + ceil(T k / nt) <= 256 + 256
// (T < 1024, k <= 16, nt = 64 above 32 tokens).
constexpr long long kMaxStreamItems = 512;
constexpr size_t kStreamCtrBytes = ((kMaxStreamItems + 4) * 4 + 255) & ~static_cast<size_t>(255);

// Token-major workspace (byte offsets): the work counter and per-item
// counters followed by the per-token row counts (one zeroed range), the
// token -> rows map [T][k], A [T*k][I] bf16, the rows' activations in expert
// order X_rows [T*k][H] bf16 and the rows' outputs [T*k][H] fp32.
struct TmLayout {
    long long items, n_zero;
    size_t tok_cnt, tok_rows, act, xp, rows, total;
};

static TmLayout tm_layout(int T, int H, int I, int N, int k) {
    TmLayout L;
    const size_t M = static_cast<size_t>(T) * k;
    L.items = ffn_max_items(T, N, k, kTmRows);
    L.n_zero = L.items + 1 + T;
    // its counters start after the weight-major kernel's region
    L.tok_cnt = kStreamCtrBytes + static_cast<size_t>(L.items + 1) * 4;
    L.tok_rows = kStreamCtrBytes + align256(static_cast<size_t>(L.n_zero) * 4);
    L.act = L.tok_rows + align256(M * 4);
    L.xp = L.act + align256(M * I * 2);
    L.rows = L.xp + align256(M * H * 2);
    L.total = L.rows + M * H * 4;
    return L;
}

// bf16 workspace.  Decode kernel (T <= 64): its counters, then A with NT
// rows per expert.  Weight-major: the counters, then A [T*k][I] bf16 (row =
// dispatch row).  Token-major: tm_layout.
size_t ffn_workspace(int T, int H, int I, int N, int k, int dtype) {
    if (dtype != MOE_DTYPE_BF16 || T <= 0) return 0;
    if (token_major(T, H)) return tm_layout(T, H, I, N, k).total;
    if (ffn_use_decode(T, k)) return ffn_decode_ctr_bytes() + static_cast<size_t>(ffn_decode_act_rows(T, N)) * I * 2;
    return kStreamCtrBytes + static_cast<size_t>(T) * k * I * 2;
}
static_assert(kStreamCtrBytes >= (MOE_MAX_EXPERTS + 4) * 4, "decode kernel counters fit the zeroed region");

// Bytes at the start of the workspace that must be zero before the first
// call (the decode and weight-major kernels' counters; the token-major
// kernels clear their own, which follow).
size_t ffn_workspace_zero_bytes(int T, int H, int N, int k, int dtype) {
    (void)H;
    (void)N;
    (void)k;
    if (dtype != MOE_DTYPE_BF16 || T <= 0) return 0;
    return kStreamCtrBytes;
}

// Items: for every active expert a, ceil(rows/NT) token chunks.  The table
// (built once per CTA in shared memory) holds, per active expert, its id,
// first row, row count and first item.
struct UnitTable {
    int* e;      // [na]
    int* row;    // [na]
    int* cnt;    // [na]
    int* pre;    // [na + 1]: exclusive prefix of chunk counts
    int na;
};

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// ---------------------------------------------------------------------------
// Two-phase streamed kernel (the bf16 path).
//
// Decode moves the active experts' weights once and does little else, so
// the kernel is cut into many small units that keep every SM streaming to
// the end.  (One unit per (chunk, I-slice) with its whole down-projection
// moves 1.5 MiB, and a batch of a few dozen active experts then splits into
// too few units to fill 152 SMs evenly.)  The FFN of every item (expert,
// token chunk) runs as
//   phase 1, S = I/128 units:  A[rows][slice] = silu(W_gate[slice] X^T) *
//            (W_up[slice] X^T), the full K = H, rounded to bf16 and stored
//            in a row-major activation buffer in the workspace;
//   phase 2, H/128 units (two per H-tile, each over half of K, when a small
//            batch would leave SMs idle): D[h-tile] = W_down[h-tile][:] A^T
//            over K = I, added as gate * D into y.
// A phase-2 unit starts once the S phase-1 units of its item have
// published their part of A (a per-item counter, release/acquire).  Units
// are handed out by a global work counter, all phase-1 units first and
// item by item, so SMs that stream faster simply take more units and the
// kernel ends within about one 192 KiB phase-2 unit of the last SM.  A unit
// is only ever taken by a running CTA, and a phase-2 unit waits only for
// phase-1 units already taken, so the waits end whatever the residency of
// the grid; a wait that outlasts kWaitLimitNs reports MOE_DEV_TIMEOUT.
// ---------------------------------------------------------------------------
template <int NT>
struct StCfg {
    static constexpr int BI = 128;                  // I-slice of a phase-1 unit (MMA M)
    static constexpr int BH = 128;                  // H-tile of a phase-2 unit (MMA M)
    static constexpr int BK = 64;                   // one 128-byte swizzle row of bf16
    static constexpr int W_BOX = 128 * 64 * 2;      // one 128 x 64 bf16 box = 16 KiB
    static constexpr int W_BYTES = 2 * W_BOX;       // gate + up (phase 1) or two K halves of W_down (phase 2)
    static constexpr int X_ATOM = NT * 128;         // NT rows of one 64-column swizzle atom
    static constexpr int X_BYTES = 2 * X_ATOM;      // phase 2 stages 128 columns of A
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int NSTAGE = NT <= 16 ? 6 : (NT <= 32 ? 5 : 4);
    static constexpr int EPI_WARPS = 8;             // two warps per TMEM lane quadrant
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int CW = NT / 2;               // token columns per epilogue warp
    static constexpr int QN = 4;                    // unit ids in flight between the warp roles
    static constexpr int NBAR = 2 * NSTAGE + 5 + 2 * QN;
    static constexpr int MISC_INTS = 8 + 64 + 8;    // tmem slot, abort flag, table size, unit ring, token list, exit flag
    static constexpr int TABLE_INTS = 6 * MOE_MAX_EXPERTS + 8;   // item table + staged active[] and offsets[]
    // dispatch rows whose token and gate are staged in shared memory at the
    // start, in one pass of the CTA's threads (batches with more rows read
    // them from global memory: a second pass would put a round trip back).
    // Batches of more than 32 tokens do not stage: measured, it cost them
    // 0.5 us even when no row was staged.
    static constexpr int RT_CAP = NT <= 16 ? 128 : (NT <= 32 ? THREADS : 0);
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + NBAR * 8 + MISC_INTS * 4 + TABLE_INTS * 4 +
                                EPI_WARPS * 32 * 8 + RT_CAP * 8;
    static constexpr uint32_t TMEM_COLS = 4 * NT;   // two accumulator slots of 2 x NT columns
    static_assert(STAGE % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256, "TMEM allocation");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(CW == 8 || CW == 16 || CW == 32, "epilogue column split");
};

__device__ __forceinline__ void item_info(const UnitTable& tb, int item, int NT, int& e, int& row0, int& nrows) {
    int lo = 0, hi = tb.na - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb.pre[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int c = item - tb.pre[lo];
    e = tb.e[lo];
    row0 = tb.row[lo] + c * NT;
    nrows = min(NT, tb.cnt[lo] - c * NT);
}

template <int NT>
__global__ void __launch_bounds__(StCfg<NT>::THREADS, 1)
    ffn_stream_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                      const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_act, const int32_t* __restrict__ offsets,
                      const int32_t* __restrict__ active, const int32_t* __restrict__ row_token,
                      const float* __restrict__ row_gate, __nv_bfloat16* __restrict__ act_g, int* counters,
                      int n_ctr, float* __restrict__ out, float* __restrict__ y_zero, long long y_elems, int H, int I,
                      int N, int fuse_combine, moe_dev_status* st, int m_rows) {
    using C = StCfg<NT>;
    constexpr int CW = C::CW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::NSTAGE * C::STAGE);
    int* misc = reinterpret_cast<int*>(bars + C::NBAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = misc + 1;
    int* s_items = misc + 2;                         // active experts, items
    volatile int* uring = misc + 4;                  // [QN] unit ids, -1 = no more work
    int* ptok = misc + 8;                            // [64] token rows of the producer's phase-1 unit
    int* table = misc + C::MISC_INTS;
    int* etok_all = table + C::TABLE_INTS;           // [EPI_WARPS][32] tokens of each epilogue warp
    float* egt_all = reinterpret_cast<float*>(etok_all + C::EPI_WARPS * 32);   // [EPI_WARPS][32] their gates
    int* s_rt = reinterpret_cast<int*>(egt_all + C::EPI_WARPS * 32);   // [RT_CAP] row -> token
    float* s_rg = reinterpret_cast<float*>(s_rt + C::RT_CAP);     // [RT_CAP] row -> gate
    const bool rt_staged = C::RT_CAP > 0 && m_rows <= C::RT_CAP;
    UnitTable tb{table, table + MOE_MAX_EXPERTS, table + 2 * MOE_MAX_EXPERTS, table + 3 * MOE_MAX_EXPERTS, 0};
    int* s_act = table + 4 * MOE_MAX_EXPERTS + 4;   // [N + 1] staged copy of active[]
    int* s_off = s_act + MOE_MAX_EXPERTS + 1;        // [N + 1] staged copy of offsets[]

    const uint32_t ring_a = smem_u32(ring);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_ACCF = 2 * C::NSTAGE, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2,
              B_QFULL = B_DRAIN + 1, B_QEMPTY = B_QFULL + C::QN;

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
        for (int i = 0; i < C::QN; ++i) {
            mbar_init(bar(B_QFULL + i), 1);
            mbar_init(bar(B_QEMPTY + i), 2);   // the MMA thread and the epilogue
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // TMEM is taken before the dependency wait (the preceding kernels hold none)
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_wg);
        tma_prefetch_desc(&tm_wu);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_act);
    }
    const int S = I / C::BI;   // phase-1 units per item
    const int MT = H / C::BH;
    const int KT2 = I / (2 * C::BK);
    int* const work_head = counters;           // next unit to hand out
    int* const item_done = counters + 1;       // phase-1 units finished, per item
    int* const zero_claim = counters + n_ctr;  // 4 KiB chunks of y handed out for zeroing
    int* const zero_done = zero_claim + 1;     // chunks of y zeroed
    int* const exit_cnt = zero_done + 1;       // CTAs that have finished
    constexpr int kZeroChunk = 1024;           // floats per chunk of y
    const int n_zchunks = (y_zero != nullptr) ? static_cast<int>((y_elems + kZeroChunk - 1) / kZeroChunk) : 0;
    pdl_wait();
    pdl_trigger();
    // the producer's first unit id is fetched while the table is built
    int first_unit = 0;
    if (warp == 0 && lane == 0) first_unit = atomicAdd(work_head, 1);
    // active[] and offsets[] in one round trip, with every row's token and
    // gate when they fit (independent loads, issued before the stores); then
    // the item table: prefix over active experts of their chunk counts
    const int n_stage = rt_staged ? max(N + 1, m_rows) : N + 1;
    for (int i = threadIdx.x; i < n_stage; i += blockDim.x) {
        int av = 0, ov = 0, rv = 0;
        float gv = 0.f;
        if (i <= N) {
            av = active[i];
            ov = offsets[i];
        }
        if (rt_staged && i < m_rows) {
            rv = row_token[i];
            gv = row_gate[i];
        }
        if (i <= N) {
            s_act[i] = av;
            s_off[i] = ov;
        }
        if (rt_staged && i < m_rows) {
            s_rt[i] = rv;
            s_rg[i] = gv;
        }
    }
    __syncthreads();
    // the last CTA to finish returns the counters to zero for the next call
    // (every CTA passes here exactly once, whatever happened before)
    int* const s_last = misc + 72;
    auto finish = [&]() {
        __syncthreads();
        if (threadIdx.x == 0) *s_last = atom_add_acq_rel_gpu(exit_cnt, 1) == static_cast<int>(gridDim.x) - 1;
        __syncthreads();
        if (*s_last)
            for (int i = threadIdx.x; i < n_ctr + 3; i += blockDim.x) counters[i] = 0;
    };
    if (warp == 2) {
        const int na = min(s_act[0], N);
        int run = 0;
        bool bad = false;
        for (int base = 0; base < na; base += 32) {
            const int a = base + lane;
            int e = 0, r0 = 0, cnt = 0, ch = 0;
            if (a < na) {
                e = s_act[1 + a];
                if (e < 0 || e >= N) e = 0;   // a corrupt list cannot index past offsets
                r0 = s_off[e];
                cnt = s_off[e + 1] - r0;
                if (r0 < 0 || cnt < 0 || r0 + cnt > m_rows) {   // rows must lie in [0, T k)
                    bad = true;
                    cnt = 0;
                }
                ch = (cnt + NT - 1) / NT;
            }
            int inc = ch;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, inc, off);
                if (lane >= off) inc += o;
            }
            if (a < na) {
                tb.e[a] = e;
                tb.row[a] = r0;
                tb.cnt[a] = cnt;
                tb.pre[a] = run + inc - ch;
            }
            run += __shfl_sync(kFull, inc, 31);
        }
        // items index the per-item counters (n_ctr - 1 of them): a dispatch
        // that would exceed them is reported and nothing is computed
        bad = __any_sync(kFull, bad) || run > n_ctr - 1;
        if (lane == 0) {
            if (bad) report(st, MOE_DEV_BAD_INDEX, run);
            tb.pre[na] = run;
            s_items[0] = bad ? 0 : na;
            s_items[1] = bad ? 0 : run;
        }
    }
    __syncthreads();
    tb.na = s_items[0];
    // With fewer than two phase-2 units per CTA (small batches) a phase-2 unit
    // covers half of K = I when the stages split evenly: its partial product
    // is added into y like a whole one, and twice the units keep more SMs
    // streaming.  (At larger batches the extra reductions into y cost more
    // than the shorter units save.)
    const int KP2 = (KT2 % 2 == 0 && s_items[1] * MT < 2 * static_cast<int>(gridDim.x)) ? 2 : 1;
    const int KT2P = KT2 / KP2;
    // units: phase 1 = [0, n1) as item * S + slice, phase 2 = [n1, n1 + n2) as
    // n1 + (item * MT + h-tile) * KP2 + K part
    const int n1 = s_items[1] * S, n_total = n1 + s_items[1] * MT * KP2;
    if (n_total == 0) {
        // no rows (or a dispatch that was rejected): y, when zeroed here, is
        // the only output
        if (y_zero != nullptr)
            for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < y_elems;
                 i += static_cast<long long>(gridDim.x) * blockDim.x)
                y_zero[i] = 0.f;
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(*tmem_slot, C::TMEM_COLS);
        }
        finish();
        return;
    }
    auto decode = [&](int u, int& item, int& sub, int& part) {
        if (u < n1) {
            item = u / S;
            sub = u - item * S;
            part = 0;
        } else {
            const int v = u - n1;
            item = v / (MT * KP2);
            const int r = v - item * MT * KP2;
            sub = r / KP2;
            part = r - sub * KP2;
        }
    };
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;   // published by the barriers since the allocation
    const int KT1 = H / C::BK;

    if (warp == 0) {
        // ---------------- TMA producer (lane 0 issues; the warp loads token lists) ----------------
        const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, pend = 0, pend_par = 0;
        bool ok = true;
        int cur = __shfl_sync(kFull, first_unit, 0);
        for (int j = 0;; ++j) {
            const bool done = cur >= n_total;
            if (lane == 0) {
                // hand the unit (or the end mark) to the MMA and epilogue warps
                const int qs = j % C::QN;
                ok = mbar_wait(bar(B_QEMPTY + qs), ((j / C::QN) & 1) ^ 1, abort_flag, st, kSiteProducerEmpty);
                if (ok) {
                    uring[qs] = done ? -1 : cur;
                    mbar_arrive(bar(B_QFULL + qs));
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok || done) break;
            // the next unit is reserved two stages before this one's last: late
            // enough that a CTA near the end of the queue holds little work an
            // idle SM could have taken, early enough to hide the counter's round
            // trip (a loop that stops early reserves nothing; the CTA stops too)
            int nxt = 0;
            const bool p1 = cur < n1;
            int item, sub, part;   // sub: I-slice or H-tile
            decode(cur, item, sub, part);
            int e, row0, nrows;
            item_info(tb, item, NT, e, row0, nrows);
            if (p1) {
                // rows past the chunk repeat its first token; their columns are never used
                for (int t = lane; t < NT; t += 32) {
                    const int r = row0 + (t < nrows ? t : 0);
                    ptok[t] = rt_staged ? s_rt[r] : row_token[r];
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (!p1) {
                    // A of this item: all S phase-1 units must have published their slices
                    const unsigned long long t0 = global_ns();
                    while (ld_acquire_gpu(item_done + item) < S ||
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
                const int n_g4 = (nrows + 3) / 4;
                const int n16 = (min(NT, max(16, (nrows + 15) & ~15))) / 16;
                const int nk = p1 ? KT1 : KT2P;
                const int kres = nk > 2 ? nk - 2 : 0;
                for (int kt = 0; kt < nk && ok; ++kt) {
                    if (kt == kres) nxt = atomicAdd(work_head, 1);
                    if (!mbar_wait(bar(B_EMPTY + stage), phase ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring_a + stage * C::STAGE;
                    const uint32_t fb = bar(B_FULL + stage);
                    if (p1) {
                        const int wrow = e * I + sub * C::BI;
                        mbar_arrive_expect_tx(fb, C::W_BYTES + n_g4 * 512);
                        tma_load_2d(dst, &tm_wg, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wu, kt * C::BK, wrow, fb, pol_w);
                        for (int g = 0; g < n_g4; ++g)
                            tma_gather4(dst + C::W_BYTES + g * 512, &tm_x, kt * C::BK, ptok[4 * g], ptok[4 * g + 1],
                                        ptok[4 * g + 2], ptok[4 * g + 3], fb, pol_x);
                    } else {
                        const int wrow = e * H + sub * C::BH;
                        const int kc = (part * KT2P + kt) * 2 * C::BK;   // first K column of this stage
                        mbar_arrive_expect_tx(fb, C::W_BYTES + 2 * n16 * 2048);
                        tma_load_2d(dst, &tm_wd, kc, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wd, kc + C::BK, wrow, fb, pol_w);
                        for (int a = 0; a < 2; ++a)
                            for (int g = 0; g < n16; ++g)
                                tma_load_2d(dst + C::W_BYTES + a * C::X_ATOM + g * 2048, &tm_act,
                                            kc + a * C::BK, row0 + 16 * g, fb, pol_x);
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
            bool ok = true;
            for (int j = 0; ok; ++j) {
                const int qs = j % C::QN;
                if (!mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteMmaFull)) break;
                const int un = uring[qs];
                mbar_arrive(bar(B_QEMPTY + qs));
                if (un < 0) break;
                const bool p1 = un < n1;
                int item, sub, part;
                decode(un, item, sub, part);
                int e, row0, nrows;
                item_info(tb, item, NT, e, row0, nrows);
                // the MMA's N is the item's row count rounded up to 16
                const uint32_t idesc = idesc_bf16_f32(128, min(NT, max(16, (nrows + 15) & ~15)));
                const int b = j & 1;
                const uint32_t acc0 = tmem + b * 2 * NT, acc1 = acc0 + NT;
                if (!mbar_wait(bar(B_ACCE + b), ((j >> 1) & 1) ^ 1, abort_flag, st, kSiteMmaTmemFree)) break;
                tc_fence_after();
                const int nk = p1 ? KT1 : KT2P;
                for (int kt = 0; kt < nk; ++kt) {
                    if (!mbar_wait(bar(B_FULL + stage), phase, abort_flag, st, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring_a + stage * C::STAGE;
                    if (p1) {
#pragma unroll
                        for (int kk = 0; kk < C::BK / 16; ++kk) {
                            const uint64_t dx = sw128_desc(a + C::W_BYTES + kk * 32);
                            const uint32_t acc = (kt | kk) != 0;
                            tc_mma_bf16(acc0, sw128_desc(a + kk * 32), dx, idesc, acc);
                            tc_mma_bf16(acc1, sw128_desc(a + C::W_BOX + kk * 32), dx, idesc, acc);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 2 * C::BK / 16; ++kk) {
                            const uint64_t dw = sw128_desc(a + (kk >> 2) * C::W_BOX + (kk & 3) * 32);
                            const uint64_t dx = sw128_desc(a + C::W_BYTES + (kk >> 2) * C::X_ATOM + (kk & 3) * 32);
                            tc_mma_bf16(acc0, dw, dx, idesc, (kt | kk) != 0);
                        }
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
        // zero y (MOE_FFN_ZERO_Y) in chunks that running warps claim, before
        // the first accumulator is ready; phase-2 units wait for all chunks
        // (zero_done), so only running CTAs ever hold a piece of y
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
        for (int j = 0;; ++j) {
            const int qs = j % C::QN;
            // every lane polls; the warp proceeds only if all lanes saw the phase complete
            bool okw = __all_sync(kFull, mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteEpiG1Done));
            const int un = okw ? uring[qs] : -1;
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (un < 0) break;   // the same value in every epilogue thread
            const bool p1 = un < n1;
            int item, sub, part;
            decode(un, item, sub, part);
            int e, row0, nrows;
            item_info(tb, item, NT, e, row0, nrows);
            const int b = j & 1;
            const uint32_t acc0 = tmem + b * 2 * NT, acc1 = acc0 + NT;
            okw = __all_sync(kFull, mbar_wait(bar(B_ACCF + b), (j >> 1) & 1, abort_flag, st, kSiteEpiG1Done));
            if (okw) {
                tc_fence_after();
                if (p1) {
                    // SwiGLU of this thread's I row for the warp's token columns -> A (bf16, row-major)
                    __nv_bfloat16* dst = act_g + static_cast<size_t>(row0) * I + sub * C::BI + row;
#pragma unroll
                    for (int c8 = 0; c8 < CW / 8; ++c8) {
                        if (c_lo + c8 * 8 >= nrows) break;   // warp-uniform
                        uint32_t g[8], u[8];
                        tmem_ld8(acc0 + lane_off + c_lo + c8 * 8, g);
                        tmem_ld8(acc1 + lane_off + c_lo + c8 * 8, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int t = c_lo + c8 * 8 + jj;
                            if (t < nrows)
                                dst[static_cast<size_t>(t) * I] =
                                    __float2bfloat16_rn(silu_mul(__uint_as_float(g[jj]), __uint_as_float(u[jj])));
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(bar(B_ACCE + b));
                    // make the stores visible to the phase-2 TMA loads of other CTAs
                    fence_proxy_async_global();
                    __threadfence();
                } else {
                    if (lane < CW) {
                        const int t = c_lo + lane;
                        etok[lane] = (t < nrows) ? (rt_staged ? s_rt[row0 + t] : row_token[row0 + t]) : 0;
                        egt[lane] = (t < nrows) ? (rt_staged ? s_rg[row0 + t] : row_gate[row0 + t]) : 0.f;
                    }
                    __syncwarp();
                    // read the accumulator in chunks of up to 16 columns; it is released right
                    // after the last read, before the last chunk's reductions
                    constexpr int CH = CW < 16 ? CW : 16;
                    const int h = sub * C::BH + row;
#pragma unroll
                    for (int c16 = 0; c16 < CW / CH; ++c16) {
                        const bool any = c_lo + c16 * CH < nrows;   // warp-uniform
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
                            const int t = c_lo + c16 * CH + jj;
                            const int js = c16 * CH + jj;
                            if (t < nrows) {
                                if (fuse_combine)
                                    atomicAdd(out + static_cast<size_t>(etok[js]) * H + h,
                                              egt[js] * __uint_as_float(vv[jj]));
                                else
                                    atomicAdd(out + static_cast<size_t>(row0 + t) * H + h, __uint_as_float(vv[jj]));
                            }
                        }
                    }
                }
            }
            // all epilogue warps pass here once per unit; a failure anywhere ends them together
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (threadIdx.x == 64) {
                if (p1) red_release_gpu_add(item_done + item, 1);
                mbar_arrive(bar(B_QEMPTY + qs));   // every epilogue thread has read the unit id
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    finish();
}

// ---------------------------------------------------------------------------
// Token-major kernel for large batches (prefill).
//
// With hundreds of rows per expert the FFN is a dense contraction, so the
// 128-row MMA operand becomes the tokens and every weight tile is used by
// 128 rows at once:
//   phase 1 unit (item = expert, chunk of <= 128 rows; I-slice s of 128):
//       D [128 x 256] = X_rows . [W_gate[s]; W_up[s]]^T over K = H, the 128
//       gate and 128 up rows of the slice loaded back to back as one N = 256
//       operand; SwiGLU -> bf16 A[rows][s*128 ...] in the workspace;
//   phase 2 unit (item, 256-row H-tile):
//       D [128 x 256] = A_rows . W_down[h-tile]^T over K = I, stored as the
//       rows' E_e(x) (each element has one writer: plain 16-byte stores).
// A prep kernel first copies the token rows into expert order (X_rows), so
// that every operand tile is one TMA box: four-row TMA gathers and fp32
// reductions into y cost about as much again as the whole contraction at
// these sizes.  A combine kernel then sums gate * E_e(x) per token over its
// rows in ascending row order (deterministic).  The work queue, the
// per-item counters and the warp roles are those of ffn_stream_kernel.
// Units are handed out expert by expert, so the chunks of one expert run
// side by side and read its weights from HBM about once.
// ---------------------------------------------------------------------------
struct PfCfg {
    static constexpr int BM = kTmRows;              // token rows per item (MMA M)
    static constexpr int BN = kTmCols;              // MMA N: gate+up of a 128-row slice, or 256 rows of H
    static constexpr int BK = 64;
    static constexpr int A_BYTES = BM * 64 * 2;     // 16 KiB
    static constexpr int B_BOX = 128 * 64 * 2;      // 16 KiB
    static constexpr int B_BYTES = 2 * B_BOX;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int NSTAGE = 4;
    static constexpr int QN = 4;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int NBAR = 2 * NSTAGE + 5 + 2 * QN;
    static constexpr int MISC_INTS = 8;             // tmem slot, abort flag, table size, unit ring
    static constexpr int TABLE_INTS = 4 * MOE_MAX_EXPERTS + 4;
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + NBAR * 8 + MISC_INTS * 4 + TABLE_INTS * 4;
    static constexpr uint32_t TMEM_COLS = 512;      // two accumulator slots of 256 columns
    static_assert(STAGE % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(SMEM <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(PfCfg::THREADS, 1)
    ffn_prefill_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                       const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_xp,
                       const __grid_constant__ CUtensorMap tm_act, const int32_t* __restrict__ offsets,
                       const int32_t* __restrict__ active, const int32_t* __restrict__ row_token,
                       __nv_bfloat16* __restrict__ act_g, int* counters, int* tok_cnt, int* tok_rows,
                       float* __restrict__ rows_out, int rows_accumulate, int H, int I, int N, int k,
                       moe_dev_status* st) {
    using C = PfCfg;
    constexpr int NT = C::BM;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::NSTAGE * C::STAGE);
    int* misc = reinterpret_cast<int*>(bars + C::NBAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = misc + 1;
    int* s_items = misc + 2;                         // active experts, items
    volatile int* uring = misc + 4;                  // [QN] unit ids, -1 = no more work
    int* table = misc + C::MISC_INTS;
    UnitTable tb{table, table + MOE_MAX_EXPERTS, table + 2 * MOE_MAX_EXPERTS, table + 3 * MOE_MAX_EXPERTS, 0};

    const uint32_t ring_a = smem_u32(ring);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_ACCF = 2 * C::NSTAGE, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2,
              B_QFULL = B_DRAIN + 1, B_QEMPTY = B_QFULL + C::QN;

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
        for (int i = 0; i < C::QN; ++i) {
            mbar_init(bar(B_QFULL + i), 1);
            mbar_init(bar(B_QEMPTY + i), 2);   // the MMA thread and the epilogue
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_wg);
        tma_prefetch_desc(&tm_wu);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_xp);
        tma_prefetch_desc(&tm_act);
    }
    const int S = I / 128, MT = H / C::BN;
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        const int na = min(active[0], N);
        int run = 0;
        for (int base = 0; base < na; base += 32) {
            const int a = base + lane;
            int e = 0, r0 = 0, cnt = 0, ch = 0;
            if (a < na) {
                e = active[1 + a];
                r0 = offsets[e];
                cnt = offsets[e + 1] - r0;
                ch = (cnt + NT - 1) / NT;
            }
            int inc = ch;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, inc, off);
                if (lane >= off) inc += o;
            }
            if (a < na) {
                tb.e[a] = e;
                tb.row[a] = r0;
                tb.cnt[a] = cnt;
                tb.pre[a] = run + inc - ch;
            }
            run += __shfl_sync(kFull, inc, 31);
        }
        if (lane == 0) {
            tb.pre[na] = run;
            s_items[0] = na;
            s_items[1] = run;
        }
    }
    __syncthreads();
    tb.na = s_items[0];
    const int n1 = s_items[1] * S, n_total = n1 + s_items[1] * MT;
    if (n_total == 0) return;
    int* const work_head = counters;
    int* const item_done = counters + 1;
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int KT1 = H / C::BK, KT2 = I / C::BK;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        const uint64_t pol_w = l2_policy_evict_last(), pol_x = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, pend = 0, pend_par = 0;
        bool ok = true;
        int cur = (lane == 0) ? atomicAdd(work_head, 1) : 0;
        cur = __shfl_sync(kFull, cur, 0);
        for (int j = 0;; ++j) {
            const bool done = cur >= n_total;
            if (lane == 0) {
                const int qs = j % C::QN;
                ok = mbar_wait(bar(B_QEMPTY + qs), ((j / C::QN) & 1) ^ 1, abort_flag, st, kSiteProducerEmpty);
                if (ok) {
                    uring[qs] = done ? -1 : cur;
                    mbar_arrive(bar(B_QFULL + qs));
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok || done) break;
            int nxt = 0;   // reserved two stages before this unit's last (as in ffn_stream_kernel)
            const bool p1 = cur < n1;
            const int v = p1 ? cur : cur - n1;
            const int item = p1 ? v / S : v / MT;
            const int sub = p1 ? v - item * S : v - item * MT;
            int e, row0, nrows;
            item_info(tb, item, NT, e, row0, nrows);
            if (lane == 0) {
                if (!p1) {
                    const unsigned long long t0 = global_ns();
                    while (ld_acquire_gpu(item_done + item) < S) {
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
                        __nanosleep(128);
                    }
                    fence_proxy_async_global();
                }
                const int nk = p1 ? KT1 : KT2;
                const int kres = nk > 2 ? nk - 2 : 0;
                for (int kt = 0; kt < nk && ok; ++kt) {
                    if (kt == kres) nxt = atomicAdd(work_head, 1);
                    if (!mbar_wait(bar(B_EMPTY + stage), phase ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring_a + stage * C::STAGE;
                    const uint32_t fb = bar(B_FULL + stage);
                    if (p1) {
                        const int wrow = e * I + sub * 128;
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                        tma_load_2d(dst, &tm_xp, kt * C::BK, row0, fb, pol_x);
                        tma_load_2d(dst + C::A_BYTES, &tm_wg, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::A_BYTES + C::B_BOX, &tm_wu, kt * C::BK, wrow, fb, pol_w);
                    } else {
                        const int wrow = e * H + sub * C::BN;
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                        tma_load_2d(dst, &tm_act, kt * C::BK, row0, fb, pol_x);
                        tma_load_2d(dst + C::A_BYTES, &tm_wd, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::A_BYTES + C::B_BOX, &tm_wd, kt * C::BK, wrow + 128, fb, pol_w);
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
            for (int i = 0; i < C::NSTAGE; ++i)
                if (pend >> i & 1u) mbar_drain(bar(B_FULL + i), pend_par >> i & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: D[128 x 256] per unit ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(128, 256);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                const int qs = j % C::QN;
                if (!mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteMmaFull)) break;
                const int un = uring[qs];
                mbar_arrive(bar(B_QEMPTY + qs));
                if (un < 0) break;
                const int b = j & 1;
                const uint32_t acc = tmem + b * C::BN;
                if (!mbar_wait(bar(B_ACCE + b), ((j >> 1) & 1) ^ 1, abort_flag, st, kSiteMmaTmemFree)) break;
                tc_fence_after();
                const int nk = (un < n1) ? KT1 : KT2;
                for (int kt = 0; kt < nk; ++kt) {
                    if (!mbar_wait(bar(B_FULL + stage), phase, abort_flag, st, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring_a + stage * C::STAGE;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc_mma_bf16(acc, sw128_desc(a + kk * 32), sw128_desc(a + C::A_BYTES + kk * 32), idesc,
                                    (kt | kk) != 0);
                    tc_commit(bar(B_EMPTY + stage));
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar(B_ACCF + b));
            }
            tc_commit(bar(B_DRAIN));
            mbar_drain(bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..9; thread = token row, warp pair splits the columns ----------------
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = q * 32 + lane;                   // row of the item
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        for (int j = 0;; ++j) {
            const int qs = j % C::QN;
            bool okw = __all_sync(kFull, mbar_wait(bar(B_QFULL + qs), (j / C::QN) & 1, abort_flag, st, kSiteEpiG1Done));
            const int un = okw ? uring[qs] : -1;
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (un < 0) break;
            const bool p1 = un < n1;
            const int v = p1 ? un : un - n1;
            const int item = p1 ? v / S : v / MT;
            const int sub = p1 ? v - item * S : v - item * MT;
            int e, row0, nrows;
            item_info(tb, item, NT, e, row0, nrows);
            const int b = j & 1;
            const uint32_t acc = tmem + b * C::BN + lane_off;
            const bool live = r < nrows;
            okw = __all_sync(kFull, mbar_wait(bar(B_ACCF + b), (j >> 1) & 1, abort_flag, st, kSiteEpiG1Done));
            if (okw) {
                tc_fence_after();
                if (p1) {
                    // this warp: I columns [64*half, 64*half + 64) of the slice; gate at +0, up at +128
                    __nv_bfloat16* dst = act_g + static_cast<size_t>(row0 + r) * I + sub * 128 + 64 * half;
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        uint32_t g[16], u[16];
                        tmem_ld16(acc + 64 * half + 16 * c16, g);
                        tmem_ld16(acc + 128 + 64 * half + 16 * c16, u);
                        tmem_ld_wait();
                        if (c16 == 3) {
                            tc_fence_before();
                            mbar_arrive(bar(B_ACCE + b));
                        }
                        if (live) {
                            uint32_t pk[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                    silu_mul(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                    silu_mul(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
                                pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
                            }
                            uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * c16);
                            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                    // the first slice of an item records its rows under their tokens for the combine
                    if (sub == 0 && half == 0 && live && tok_cnt != nullptr) {
                        const int t = row_token[row0 + r];
                        tok_rows[static_cast<size_t>(t) * k + atomicAdd(tok_cnt + t, 1)] = row0 + r;
                    }
                    fence_proxy_async_global();
                    __threadfence();
                } else {
                    // this warp: H columns [128*half, 128*half + 128) of the 256-row tile; every
                    // element of rows_out has exactly this one writer
                    float* dst = rows_out + static_cast<size_t>(row0 + r) * H + sub * C::BN + 128 * half;
#pragma unroll 1
                    for (int c16 = 0; c16 < 8; ++c16) {
                        uint32_t d[16];
                        tmem_ld16(acc + 128 * half + 16 * c16, d);
                        tmem_ld_wait();
                        if (c16 == 7) {
                            tc_fence_before();
                            mbar_arrive(bar(B_ACCE + b));
                        }
                        if (live) {
                            float4* d4 = reinterpret_cast<float4*>(dst + 16 * c16);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float4 v = make_float4(__uint_as_float(d[4 * i]), __uint_as_float(d[4 * i + 1]),
                                                       __uint_as_float(d[4 * i + 2]), __uint_as_float(d[4 * i + 3]));
                                if (rows_accumulate) {
                                    const float4 o = d4[i];
                                    v.x += o.x;
                                    v.y += o.y;
                                    v.z += o.z;
                                    v.w += o.w;
                                }
                                d4[i] = v;
                            }
                        }
                    }
                }
            }
            if (!named_sync_and(C::EPI_THREADS, okw)) break;
            if (threadIdx.x == 64) {
                if (p1) red_release_gpu_add(item_done + item, 1);
                mbar_arrive(bar(B_QEMPTY + qs));
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Token-major path, before the FFN kernel: clears the work, item and token
// counters and copies every dispatch row's activations into expert order,
// X_rows[r] = x[row_token[r]] (16-byte vectors, one warp per row).
__global__ void __launch_bounds__(256) ffn_tm_prep_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ row_token,
                                                          const int32_t* __restrict__ offsets, int N, int H,
                                                          uint4* __restrict__ xp, int* zero, int n_zero) {
    pdl_wait();
    pdl_trigger();
    const int gtid = blockIdx.x * 256 + threadIdx.x, nthr = gridDim.x * 256;
    for (int i = gtid; i < n_zero; i += nthr) zero[i] = 0;
    const int M = offsets[N];
    const int v = H / 8;
    const int lane = threadIdx.x & 31;
    // one warp per row, a row's 16-byte loads issued 8 at a time before the stores
    for (int r = gtid >> 5; r < M; r += nthr >> 5) {
        const uint4* src = x + static_cast<size_t>(row_token[r]) * v;
        uint4* d = xp + static_cast<size_t>(r) * v;
        for (int c0 = lane; c0 < v; c0 += 32 * 8) {
            uint4 q[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int c = c0 + 32 * m;
                q[m] = (c < v) ? src[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int c = c0 + 32 * m;
                if (c < v) d[c] = q[m];
            }
        }
    }
}

// Token-major path, after the FFN kernel: y[t] = (y[t] or 0) + sum over the
// token's rows, in ascending row order, of gate * E_e(x_t).  Per token, warp
// 0 reads the row list in one round trip and ranks the rows with shuffles
// (a token's rows are distinct), then every thread issues all of its row
// loads before adding them up in that order.
template <int KMAX>
__global__ void __launch_bounds__(256) ffn_tm_combine_kernel(const float* __restrict__ rows,
                                                             const int* __restrict__ tok_cnt,
                                                             const int* __restrict__ tok_rows,
                                                             const float* __restrict__ row_gate, int T, int H,
                                                             int k, int zero_y, float* __restrict__ y) {
    __shared__ int srow[KMAX];
    __shared__ float sg[KMAX];
    __shared__ int sn;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H4 = H / 4;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (warp == 0) {
            const int n = min(tok_cnt[t], k);
            const int v = (lane < k) ? tok_rows[static_cast<size_t>(t) * k + lane] : 0;
            int rank = 0;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const int vj = __shfl_sync(kFull, v, j);
                if (j < n && vj < v) ++rank;
            }
            if (lane < n) {
                srow[rank] = v;
                sg[rank] = row_gate[v];
            }
            if (lane == 0) sn = n;
        }
        __syncthreads();
        const int n = sn;
        float4* yt = reinterpret_cast<float4*>(y + static_cast<size_t>(t) * H);
        for (int hb = threadIdx.x; hb < H4; hb += 2 * 256) {
            float4 v[KMAX][2];
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int h4 = hb + 256 * m;
                    v[i][m] = (i < n && h4 < H4) ? reinterpret_cast<const float4*>(rows + static_cast<size_t>(srow[i]) * H)[h4]
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int h4 = hb + 256 * m;
                if (h4 >= H4) break;
                float4 acc = zero_y ? make_float4(0.f, 0.f, 0.f, 0.f) : yt[h4];
#pragma unroll
                for (int i = 0; i < KMAX; ++i) {
                    if (i < n) {
                        acc.x = fmaf(sg[i], v[i][m].x, acc.x);
                        acc.y = fmaf(sg[i], v[i][m].y, acc.y);
                        acc.z = fmaf(sg[i], v[i][m].z, acc.z);
                        acc.w = fmaf(sg[i], v[i][m].w, acc.w);
                    }
                }
                yt[h4] = acc;
            }
        }
        __syncthreads();   // the row list is read by every thread before the next token's
    }
}

// ---------------------------------------------------------------------------
// Host side of the tensor-core path.
// ---------------------------------------------------------------------------
__global__ void zero_kernel(float* p, long long n, int* c, int nc);

// Clears p[0, n) (fp32) and c[0, nc) (int32) in one launch.
static cudaError_t launch_zero(float* p, long long n, cudaStream_t s, int* c = nullptr, int nc = 0) {
    int grid = static_cast<int>((n / 4 + 255) / 256);
    grid = grid < 1 ? 1 : (grid > 1024 ? 1024 : grid);
    return launch_pdl(zero_kernel, dim3(grid), dim3(256), 0, s, p, n, c, nc);
}

template <int NT>
static cudaError_t run_stream(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                              int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                              const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                              cudaStream_t s) {
    using C = StCfg<NT>;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    const long long M = static_cast<long long>(T) * k;
    const long long items = ffn_max_items(T, N, k, NT);
    // counters: work head, per-item counters, then zero_claim, zero_done and
    // exit_cnt; zero before the first call, and returned to zero by every call
    if (items > kMaxStreamItems) return cudaErrorInvalidValue;
    int* counters = static_cast<int*>(ws);
    __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + kStreamCtrBytes);
    float* y_zero = (fuse && (flags & MOE_FFN_ZERO_Y)) ? out : nullptr;
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x, tm_act;
    if (!make_tmap(&tm_wg, wg, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wu, wu, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wd, wd, I, static_cast<uint64_t>(N) * H, 64, 128) ||
        !make_tmap(&tm_x, x, H, static_cast<uint64_t>(T), 64, 1) ||
        !make_tmap(&tm_act, act, I, static_cast<uint64_t>(M), 64, 16))
        return cudaErrorInvalidValue;
    // the attribute is set once per device, on the first (uncaptured) call
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int devi = 0;
    cudaGetDevice(&devi);
    if (devi < 0 || devi >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[devi]) {
        cudaError_t ae =
            cudaFuncSetAttribute(ffn_stream_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (ae != cudaSuccess) return ae;
        attr_set[devi] = true;
    }
    const long long max_units = items * (I / C::BI + H / C::BH);
    int grid = sm_count();
    if (max_units < grid) grid = static_cast<int>(max_units > 0 ? max_units : 1);
    return launch_pdl(ffn_stream_kernel<NT>, dim3(grid), dim3(C::THREADS), C::SMEM, s, tm_wg, tm_wu, tm_wd, tm_x,
                      tm_act, offsets, active, row_token, row_gate, act, counters, static_cast<int>(items + 1), out,
                      y_zero, static_cast<long long>(T) * H, H, I, N, fuse ? 1 : 0, st, static_cast<int>(M));
}

static cudaError_t run_tokmajor(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                                int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                                const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                                cudaStream_t s) {
    using C = PfCfg;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    const long long M = static_cast<long long>(T) * k;
    const TmLayout Lw = tm_layout(T, H, I, N, k);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int* counters = reinterpret_cast<int*>(base + kStreamCtrBytes);   // tok_cnt follows the item counters
    int* tok_cnt = reinterpret_cast<int*>(base + Lw.tok_cnt);
    int* tok_rows = reinterpret_cast<int*>(base + Lw.tok_rows);
    __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(base + Lw.act);
    void* xp = base + Lw.xp;
    float* rows = reinterpret_cast<float*>(base + Lw.rows);
    const int sms = sm_count();
    cudaError_t e = launch_pdl(ffn_tm_prep_kernel, dim3(4 * sms), dim3(256), 0, s, static_cast<const uint4*>(x),
                               row_token, offsets, N, H, static_cast<uint4*>(xp), counters,
                               static_cast<int>(Lw.n_zero));
    if (e != cudaSuccess) return e;
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_xp, tm_act;
    if (!make_tmap(&tm_wg, wg, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wu, wu, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wd, wd, I, static_cast<uint64_t>(N) * H, 64, 128) ||
        !make_tmap(&tm_xp, xp, H, static_cast<uint64_t>(M), 64, 128) ||
        !make_tmap(&tm_act, act, I, static_cast<uint64_t>(M), 64, 128))
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int devi = 0;
    cudaGetDevice(&devi);
    if (devi < 0 || devi >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[devi]) {
        cudaError_t ae = cudaFuncSetAttribute(ffn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (ae != cudaSuccess) return ae;
        attr_set[devi] = true;
    }
    const long long max_units = Lw.items * (I / 128 + H / C::BN);
    int grid = sms;
    if (max_units < grid) grid = static_cast<int>(max_units > 0 ? max_units : 1);
    e = launch_pdl(ffn_prefill_kernel, dim3(grid), dim3(C::THREADS), C::SMEM, s, tm_wg, tm_wu, tm_wd, tm_xp, tm_act,
                   offsets, active, row_token, act, counters, fuse ? tok_cnt : static_cast<int*>(nullptr), tok_rows,
                   fuse ? rows : out, fuse ? 0 : 1, H, I, N, k, st);
    if (e != cudaSuccess || !fuse) return e;
    const int cgrid = T < 8 * sms ? T : 8 * sms;
    if (k <= 8)
        return launch_pdl(ffn_tm_combine_kernel<8>, dim3(cgrid), dim3(256), 0, s, static_cast<const float*>(rows),
                          static_cast<const int*>(tok_cnt), static_cast<const int*>(tok_rows), row_gate, T, H, k,
                          (flags & MOE_FFN_ZERO_Y) ? 1 : 0, out);
    return launch_pdl(ffn_tm_combine_kernel<MOE_MAX_RANKS>, dim3(cgrid), dim3(256), 0, s,
                      static_cast<const float*>(rows), static_cast<const int*>(tok_cnt),
                      static_cast<const int*>(tok_rows), row_gate, T, H, k, (flags & MOE_FFN_ZERO_Y) ? 1 : 0, out);
}

cudaError_t launch_ffn_bf16(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                            int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                            const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                            cudaStream_t s) {
    // batches with many rows per expert run token-major on the tensor cores
    if (token_major(T, H))
        return run_tokmajor(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, ws, st, s);
    // decode batches: the all-token kernel (ffn_decode.cu)
    if (ffn_use_decode(T, k))
        return launch_ffn_decode(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, nullptr, flags,
                                 out, ws, st, s);
    return run_stream<kStreamNT>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, ws,
                                 st, s);
}

// ---------------------------------------------------------------------------
// fp32 CUDA-core path: one CTA per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ffn_f32_kernel(const float* __restrict__ x, const float* __restrict__ wg,
                                                      const float* __restrict__ wu, const float* __restrict__ wd,
                                                      int H, int I, int N, const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ row_token,
                                                      const float* __restrict__ row_gate, int fuse,
                                                      float* __restrict__ out) {
    extern __shared__ float sh[];
    float* xs = sh;       // [H]
    float* as = sh + H;   // [I]
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    if (row >= offsets[N]) return;
    // expert of this row: offsets is ascending; binary search
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int tok = row_token[row];
    for (int h = threadIdx.x; h < H; h += blockDim.x) xs[h] = x[static_cast<size_t>(tok) * H + h];
    __syncthreads();
    for (int i = threadIdx.x; i < I; i += blockDim.x) {
        const float* g = wg + (static_cast<size_t>(e) * I + i) * H;
        const float* u = wu + (static_cast<size_t>(e) * I + i) * H;
        float a = 0.f, b = 0.f;
        for (int h = 0; h < H; ++h) {
            a = fmaf(g[h], xs[h], a);
            b = fmaf(u[h], xs[h], b);
        }
        as[i] = silu_mul(a, b);
    }
    __syncthreads();
    const float gate = row_gate[row];
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float* d = wd + (static_cast<size_t>(e) * H + h) * I;
        float acc = 0.f;
        for (int i = 0; i < I; ++i) acc = fmaf(d[i], as[i], acc);
        if (fuse) atomicAdd(out + static_cast<size_t>(tok) * H + h, gate * acc);
        else out[static_cast<size_t>(row) * H + h] = acc;
    }
}

__global__ void zero_kernel(float* p, long long n, int* c, int nc) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x * 256 + threadIdx.x; i < nc; i += 256 * gridDim.x) c[i] = 0;
    const long long n4 = n / 4;
    float4* p4 = reinterpret_cast<float4*>(p);
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n4; i += 256ll * gridDim.x)
        p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = n4 * 4 + blockIdx.x * 256ll + threadIdx.x; i < n; i += 256ll * gridDim.x) p[i] = 0.f;
}

cudaError_t launch_ffn_f32(const float* x, const float* wg, const float* wu, const float* wd, int T, int H, int I,
                           int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                           const int32_t* active, uint32_t flags, float* out, moe_dev_status* st, cudaStream_t s) {
    (void)active;
    (void)st;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    if (fuse && (flags & MOE_FFN_ZERO_Y)) {
        cudaError_t e = launch_zero(out, static_cast<long long>(T) * H, s);
        if (e != cudaSuccess) return e;
    }
    const int Mmax = T * k;
    if (Mmax == 0) return cudaGetLastError();
    const size_t smem = sizeof(float) * static_cast<size_t>(H + I);
    if (smem > static_cast<size_t>(kFfnF32MaxSmem)) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        // raised once per device to the largest size and never lowered, so
        // that calls of different sizes from several host threads cannot
        // undo each other's setting
        static std::atomic<bool> attr_set[64] = {};
        int devi = 0;
        cudaError_t e = cudaGetDevice(&devi);
        if (e != cudaSuccess) return e;
        if (devi < 0 || devi >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[devi]) {
            e = cudaFuncSetAttribute(ffn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFfnF32MaxSmem);
            if (e != cudaSuccess) return e;
            attr_set[devi] = true;
        }
    }
    return launch_pdl(ffn_f32_kernel, dim3(Mmax), dim3(256), smem, s, x, wg, wu, wd, H, I, N, offsets, row_token,
                      row_gate, fuse ? 1 : 0, out);
}

// ---------------------------------------------------------------------------
// Deterministic combine: y[t] = sum over slots (in slot order) of gate * row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ rows_out,
                                                      const int32_t* __restrict__ slot_row,
                                                      const float* __restrict__ slot_gate, int T, int H, int k,
                                                      float* __restrict__ y) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int h = blockIdx.x * 256 + threadIdx.x;
    if (t >= T || h >= H) return;
    float acc = 0.f;
    for (int r = 0; r < k; ++r) {
        const int row = slot_row[static_cast<size_t>(t) * k + r];
        if (row >= 0) acc = fmaf(slot_gate[static_cast<size_t>(t) * k + r], rows_out[static_cast<size_t>(row) * H + h], acc);
    }
    y[static_cast<size_t>(t) * H + h] = acc;
}

cudaError_t launch_combine(const float* rows_out, const int32_t* slot_row, const float* slot_gate, int T, int H,
                           int k, float* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    dim3 grid((H + 255) / 256, T);
    return launch_pdl(combine_kernel, grid, dim3(256), 0, s, rows_out, slot_row, slot_gate, T, H, k, y);
}

}  // namespace moe
