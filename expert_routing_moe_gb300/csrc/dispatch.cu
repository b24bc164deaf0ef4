// dispatch.cu -- expert-sorted permutation and the capacity-bounded dispatch.
//
// Token sets I_j and the straggler bound: "MACS: Modality-Aware Capacity
// Scaling for Efficient Multimodal MoE Inference", sec. 3.1 Eqs. (2)-(3);
// weighted load: sec. 3.2 Eq. (6); overflow handling (reroute locally, else
// drop): Fig. 1 and the sec. 3.4 summary in the introduction.
//
// Permutation: rows ordered by (expert asc, token asc).  Because a token
// holds an expert at most once, a row's position is the expert's start plus
// the number of earlier tokens holding that expert; that count comes from a
// per-expert presence bitmap over the tokens of a 1024-token block and
// population counts, so the result is deterministic without any sort.
//
// Capacity: loads are integers in 2^-24 units (exact, order-free sums).  Each
// expert's candidates are sorted by (gate desc, token asc) with a bitonic sort
// in shared memory and admitted while the running load stays within C.
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "permute.cuh"

namespace moe {

constexpr uint8_t kPending = 255;

static inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct DispatchWs {
    int32_t* blk_start;   // [nblk][N]
    // capacity mode only
    unsigned long long* S;
    int32_t* cnt1;        // [N]
    int32_t* cnt2;        // [N]
    uint32_t* bucket1;    // [N][T]
    uint32_t* bucket2;    // [N][T]
    long long* load;      // [N]
    uint8_t* status;      // [T][k]
    int32_t* wids;        // [T][k]
    float* wgates;        // [T][k]
    size_t zero_bytes;    // bytes from S to the end of cnt2 (cleared per call)
    const int8_t* bias;   // [N] modality bias m_j, or null (static capacity)
    const float* r_v;     // [1] effective visual ratio, with bias
};

// Tokens per block of the multi-block permutation (below).
constexpr int kMbBlk = 256;

static size_t carve(DispatchWs* w, void* base, int T, int N, int k, bool capped) {
    const int nblk = (T + kMbBlk - 1) / kMbBlk;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    size_t o_blk = take(sizeof(int32_t) * static_cast<size_t>(nblk > 0 ? nblk : 1) * N);
    size_t o_S = 0, o_c1 = 0, o_c2 = 0, o_b1 = 0, o_b2 = 0, o_ld = 0, o_st = 0, o_id = 0, o_g = 0;
    if (capped) {
        o_S = take(sizeof(unsigned long long));
        o_c1 = take(sizeof(int32_t) * N);
        o_c2 = take(sizeof(int32_t) * N);
        o_b1 = take(sizeof(uint32_t) * static_cast<size_t>(N) * (T > 0 ? T : 1));
        o_b2 = take(sizeof(uint32_t) * static_cast<size_t>(N) * (T > 0 ? T : 1));
        o_ld = take(sizeof(long long) * N);
        o_st = take(static_cast<size_t>(T > 0 ? T : 1) * k);
        o_id = take(sizeof(int32_t) * static_cast<size_t>(T > 0 ? T : 1) * k);
        o_g = take(sizeof(float) * static_cast<size_t>(T > 0 ? T : 1) * k);
    }
    if (w != nullptr) {
        char* b = static_cast<char*>(base);
        w->blk_start = reinterpret_cast<int32_t*>(b + o_blk);
        if (capped) {
            w->S = reinterpret_cast<unsigned long long*>(b + o_S);
            w->cnt1 = reinterpret_cast<int32_t*>(b + o_c1);
            w->cnt2 = reinterpret_cast<int32_t*>(b + o_c2);
            w->bucket1 = reinterpret_cast<uint32_t*>(b + o_b1);
            w->bucket2 = reinterpret_cast<uint32_t*>(b + o_b2);
            w->load = reinterpret_cast<long long*>(b + o_ld);
            w->status = reinterpret_cast<uint8_t*>(b + o_st);
            w->wids = reinterpret_cast<int32_t*>(b + o_id);
            w->wgates = reinterpret_cast<float*>(b + o_g);
            w->zero_bytes = o_b1 - o_S;
        }
    }
    return off;
}

size_t dispatch_workspace(int T, int N, int k, int R, bool capped) {
    (void)R;
    return carve(nullptr, nullptr, T, N, k, capped);
}

// Single-block permutation (T <= 1024): presence, counts, scan and rows in one launch.
__global__ void __launch_bounds__(kBlk) permute_single_kernel(const int32_t* __restrict__ ids,
                                                              const float* __restrict__ gates, int ld, int T, int N,
                                                              int k, int32_t* counts, int32_t* offsets,
                                                              int32_t* row_token, float* row_gate, int32_t* active,
                                                              int32_t* out_ids, float* out_gates,
                                                              int32_t* slot_row, moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t bits[MOE_MAX_EXPERTS * kWordsPerBlk];
    __shared__ int cnt[MOE_MAX_EXPERTS];
    __shared__ int start[MOE_MAX_EXPERTS];
    const int nw = (T + 31) / 32;
    presence_bits(ids, ld, T, N, k, 0, nw, bits, st);
    for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = block_count(bits, e, nw);
    __syncthreads();
    scan_experts(cnt, N, counts, offsets, active, start);
    __syncthreads();
    write_rows(ids, gates, ld, T, N, k, 0, nw, bits, start, row_token, row_gate, out_ids, out_gates, slot_row);
}

// Multi-block permutation over blocks of kMbBlk tokens (more, smaller
// blocks keep more SMs busy at prefill sizes).  The presence bitmap of a
// block has kMbWords words per expert, stored with a stride of kMbWords + 1
// so that lanes reading different experts' words rarely share a bank.
constexpr int kMbWords = kMbBlk / 32;
constexpr int kMbStride = kMbWords + 1;

// Marks bit (t mod 32) of word (t / 32) of expert e for every slot of token t
// of block b holding e.
__device__ __forceinline__ void mb_presence(const int32_t* __restrict__ ids, int ld, int T, int N, int k, int b,
                                            uint32_t* bits, moe_dev_status* st) {
    for (int i = threadIdx.x; i < N * kMbStride; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    const int t = b * kMbBlk + threadIdx.x;
    if (t < T) {
        for (int r = 0; r < k; ++r) {
            const int e = ids[static_cast<size_t>(t) * ld + r];
            if (e >= N && st != nullptr) report(st, MOE_DEV_BAD_INDEX, e);
            if (e >= 0 && e < N) atomicOr(&bits[e * kMbStride + (threadIdx.x >> 5)], 1u << (threadIdx.x & 31));
        }
    }
    __syncthreads();
}

// Pass 1: per-block expert counts.
__global__ void __launch_bounds__(kMbBlk) permute_count_kernel(const int32_t* __restrict__ ids, int ld, int T, int N,
                                                               int k, int32_t* __restrict__ blk_cnt,
                                                               moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t bits[MOE_MAX_EXPERTS * kMbStride];
    mb_presence(ids, ld, T, N, k, blockIdx.x, bits, st);
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kMbWords; ++w) c += __popc(bits[e * kMbStride + w]);
        blk_cnt[static_cast<size_t>(blockIdx.x) * N + e] = c;
    }
}

// Pass 2 (one CTA of 1024 threads): totals, offsets, active list; blk_cnt
// becomes the absolute start row of each (block, expert).  One warp per
// expert scans its block counts, 32 blocks per lane pass (all loads issued
// first); integer sums, so the order of the adds does not matter.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int nblk, int N, int32_t* __restrict__ blk_cnt,
                                                            int32_t* counts, int32_t* offsets, int32_t* active) {
    pdl_wait();
    pdl_trigger();
    __shared__ int tot[MOE_MAX_EXPERTS];
    __shared__ int start[MOE_MAX_EXPERTS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int e = warp; e < N; e += nwarps) {
        int run = 0;
        for (int b0 = 0; b0 < nblk; b0 += 32) {
            const int b = b0 + lane;
            const int c = (b < nblk) ? blk_cnt[static_cast<size_t>(b) * N + e] : 0;
            int inc = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, inc, off);
                if (lane >= off) inc += o;
            }
            if (b < nblk) blk_cnt[static_cast<size_t>(b) * N + e] = run + inc - c;
            run += __shfl_sync(kFull, inc, 31);
        }
        if (lane == 0) tot[e] = run;
    }
    __syncthreads();
    scan_experts(tot, N, counts, offsets, active, start);
    __syncthreads();
    for (int i = threadIdx.x; i < nblk * N; i += blockDim.x) blk_cnt[i] += start[i % N];
}

// Pass 3: rows of each block.  pre[e][w] = start of expert e in this block
// plus the set bits of its words before w, so a slot's row is pre[e][w] plus
// the set bits below its token in word w: (expert, token) order, as in the
// single-block kernel.
__global__ void __launch_bounds__(kMbBlk) permute_rows_kernel(const int32_t* __restrict__ ids,
                                                              const float* __restrict__ gates, int ld, int T, int N,
                                                              int k, const int32_t* __restrict__ blk_start,
                                                              int32_t* row_token, float* row_gate, int32_t* out_ids,
                                                              float* out_gates, int32_t* slot_row,
                                                              moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t bits[MOE_MAX_EXPERTS * kMbStride];
    __shared__ int pre[MOE_MAX_EXPERTS * kMbStride];
    mb_presence(ids, ld, T, N, k, blockIdx.x, bits, nullptr);
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int run = blk_start[static_cast<size_t>(blockIdx.x) * N + e];
#pragma unroll
        for (int w = 0; w < kMbWords; ++w) {
            pre[e * kMbStride + w] = run;
            run += __popc(bits[e * kMbStride + w]);
        }
    }
    __syncthreads();
    const int t = blockIdx.x * kMbBlk + threadIdx.x;
    if (t >= T) return;
    const int w0 = threadIdx.x >> 5;
    const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
    for (int r = 0; r < k; ++r) {
        const size_t si = static_cast<size_t>(t) * ld + r;
        const size_t so = static_cast<size_t>(t) * k + r;
        const int e = ids[si];
        const float g = gates[si];
        int row = -1;
        if (e >= 0 && e < N) {
            row = pre[e * kMbStride + w0] + __popc(bits[e * kMbStride + w0] & below);
            row_token[row] = t;
            row_gate[row] = g;
        }
        if (slot_row) slot_row[so] = row;
        if (out_ids) out_ids[so] = (row >= 0) ? e : -1;
        if (out_gates) out_gates[so] = (row >= 0) ? g : 0.f;
    }
    (void)st;
}

static cudaError_t launch_permute(const int32_t* ids, const float* gates, int ld, int T, int N, int k,
                                  int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_gate,
                                  int32_t* active, int32_t* out_ids, float* out_gates, int32_t* slot_row,
                                  int32_t* blk_start, moe_dev_status* st, cudaStream_t s) {
    if (T <= kBlk) {
        const int threads = T <= 128 ? 128 : (T + 31) / 32 * 32;
        return launch_pdl(permute_single_kernel, dim3(1), dim3(threads), 0, s, ids, gates, ld, T, N, k, counts,
                          offsets, row_token, row_gate, active, out_ids, out_gates, slot_row, st);
    }
    const int nblk = (T + kMbBlk - 1) / kMbBlk;
    cudaError_t e = launch_pdl(permute_count_kernel, dim3(nblk), dim3(kMbBlk), 0, s, ids, ld, T, N, k, blk_start, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, s, nblk, N, blk_start, counts, offsets, active);
    if (e != cudaSuccess) return e;
    return launch_pdl(permute_rows_kernel, dim3(nblk), dim3(kMbBlk), 0, s, ids, gates, ld, T, N, k,
                      static_cast<const int32_t*>(blk_start), row_token, row_gate, out_ids, out_gates, slot_row, st);
}

// ---------------------------------------------------------------------------
// Capacity mode
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long fixed_weight(float w) {
    return static_cast<long long>(rintf(__fmul_rn(w, 16777216.0f)));
}

__device__ __forceinline__ long long capacity_value(unsigned long long S, int k, float gamma, int N) {
    const double a = __dmul_rn(static_cast<double>(S), static_cast<double>(k));
    const double b = __dmul_rn(a, static_cast<double>(gamma));
    return static_cast<long long>(floor(__ddiv_rn(b, static_cast<double>(N))));
}

// Capacity of expert e.  "MACS" sec. 3.3 scales each expert's capacity by its
// modality (m_e = +1 visual, -1 text, 0 shared) and the batch's effective
// visual ratio R_v; the page stops before the formula.  Reading:
// C_e = floor(c * (1 + m_e * (R_v - 1/2))), c the unfloored static capacity,
// each operation rounded on its own in this order.  An out-of-range bias or
// ratio is reported and treated as m_e = 0.
__device__ __forceinline__ long long capacity_of(const DispatchWs& w, int e, int k, float gamma, int N,
                                                 moe_dev_status* st) {
    const unsigned long long S = *w.S;
    if (w.bias == nullptr) return capacity_value(S, k, gamma, N);
    const int m = w.bias[e];
    const float rv = *w.r_v;
    if (m < -1 || m > 1) {
        report(st, MOE_DEV_BAD_INDEX, m);
        return capacity_value(S, k, gamma, N);
    }
    if (!(rv >= 0.f && rv <= 1.f)) {
        report(st, MOE_DEV_NONFINITE, e);
        return capacity_value(S, k, gamma, N);
    }
    const double c = __ddiv_rn(__dmul_rn(__dmul_rn(static_cast<double>(S), static_cast<double>(k)),
                                         static_cast<double>(gamma)),
                               static_cast<double>(N));
    const double scale = __dadd_rn(1.0, __dmul_rn(static_cast<double>(m), __dsub_rn(static_cast<double>(rv), 0.5)));
    return static_cast<long long>(floor(__dmul_rn(c, scale)));
}

// Phase-1 bucketing: fixed-point weights, total S, copies of the slots, and
// each slot appended to its expert's bucket (order fixed later by the keys).
// S is summed per block (one global atomic per block); a token's k slots are
// loaded together; slots of one warp that name the same expert reserve their
// bucket positions with one atomic.
__global__ void __launch_bounds__(128) cap_bucket_kernel(const int32_t* __restrict__ ids,
                                                         const float* __restrict__ gates, int ld, int T, int N,
                                                         int k, const float* __restrict__ token_w, DispatchWs w,
                                                         moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ unsigned long long sS;
    if (threadIdx.x == 0) sS = 0ull;
    __syncthreads();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    unsigned long long wq = 0ull;
    int ev[MOE_MAX_RANKS];
    float gv[MOE_MAX_RANKS];
    if (t < T) {
        float wt = token_w ? token_w[t] : 1.0f;
        if (!isfinite(wt) || wt < 0.f) {
            report(st, MOE_DEV_NONFINITE, t);
            wt = 0.f;
        }
        wq = static_cast<unsigned long long>(fixed_weight(wt));
#pragma unroll
        for (int r = 0; r < MOE_MAX_RANKS; ++r) {
            if (r < k) {
                ev[r] = ids[static_cast<size_t>(t) * ld + r];
                gv[r] = gates[static_cast<size_t>(t) * ld + r];
            }
        }
    }
    for (int off = 16; off >= 1; off >>= 1) wq += __shfl_xor_sync(kFull, wq, off);
    if (lane == 0) atomicAdd(&sS, wq);
#pragma unroll
    for (int r = 0; r < MOE_MAX_RANKS; ++r) {
        if (r >= k) break;
        int e = -1;
        if (t < T) {
            const size_t so = static_cast<size_t>(t) * k + r;
            e = ev[r];
            w.wids[so] = e;
            w.wgates[so] = gv[r];
            w.status[so] = kPending;
            if (e < 0 || e >= N) {
                report(st, MOE_DEV_BAD_INDEX, e);
                w.status[so] = MOE_SLOT_DROPPED;
                w.wids[so] = -1;
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0) {
            const int leader = __ffs(peers) - 1;
            int pos0 = 0;
            if (lane == leader) pos0 = atomicAdd(&w.cnt1[e], __popc(peers));
            const int pos = __shfl_sync(peers, pos0, leader) + __popc(peers & ((1u << lane) - 1u));
            if (pos >= T) {   // only possible if a token holds the same expert twice
                report(st, MOE_DEV_BAD_INDEX, e);
            } else {
                w.bucket1[static_cast<size_t>(e) * T + pos] = static_cast<uint32_t>(t) * 16u + static_cast<uint32_t>(r);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(w.S, sS);
}

// One CTA per expert: admit its candidates in (gate desc, token asc) order
// while load + running weight <= C (a strict prefix).  `round` < 0 is phase 1
// (candidates are the expert's own slots); round i >= 0 admits overflow
// offers as rerouted.
//
// The prefix is found without sorting everything.  Keys (~gate bits, token,
// slot) ascend in admission order.  If all candidates fit, all are admitted.
// Otherwise a weight histogram over 1024 bins of the key range locates the
// one bin b* in which the running weight crosses C: every candidate in an
// earlier bin is admitted, every one in a later bin is not, and only b*'s
// candidates are sorted (bitonic) and admitted in exact order.  The outcome
// equals that of sorting all candidates.
constexpr int kCapBins = 1024;
constexpr int kCapPer = kCapacityMaxT / 1024;   // candidates per thread at most
// dynamic shared memory of cap_admit_kernel at the largest batch: the sort
// keys padded to a power of two, then one fp32 weight per token
constexpr int kCapAdmitMaxSmem = kCapacityMaxT * 8 + kCapacityMaxT * 4;
static_assert(kCapAdmitMaxSmem <= 227 * 1024, "cap_admit shared memory");

__device__ __forceinline__ float cap_weight(const float* token_w, int t) {
    float wt = token_w ? token_w[t] : 1.0f;
    return (!isfinite(wt) || wt < 0.f) ? 0.f : wt;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long s = 0ull;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
    return s;
}

__global__ void __launch_bounds__(1024) cap_admit_kernel(const float* __restrict__ gates, int ld, int T, int N,
                                                         int k, float gamma, const float* __restrict__ token_w,
                                                         int round, DispatchWs w, moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ unsigned long long keys[];       // [P2(T)] candidate keys, then [T] float weights
    __shared__ unsigned long long hist[kCapBins];
    __shared__ unsigned long long red[32];
    __shared__ unsigned long long s_kmin, s_kmax, s_adm;
    __shared__ long long s_excl;
    __shared__ int s_bstar, s_m;
    int P2T = 1;
    while (P2T < T) P2T <<= 1;
    float* wts = reinterpret_cast<float*>(keys + P2T);
    const int e = blockIdx.x;
    const int n = min((round < 0) ? w.cnt1[e] : w.cnt2[e], T);
    const uint32_t* bucket = ((round < 0) ? w.bucket1 : w.bucket2) + static_cast<size_t>(e) * T;
    const long long C = capacity_of(w, e, k, gamma, N, st);
    const long long base = (round < 0) ? 0ll : w.load[e];
    auto admit = [&](uint32_t tr) {
        const size_t so = static_cast<size_t>(tr >> 4) * k + (tr & 15u);
        if (round < 0) {
            w.status[so] = MOE_SLOT_KEPT;
        } else {
            w.status[so] = MOE_SLOT_REROUTED;
            w.wids[so] = e;
        }
    };
    // candidates: keys and weights (independent loads, batched per thread)
    unsigned long long tot = 0ull, kmin = ~0ull, kmax = 0ull;
#pragma unroll
    for (int j = 0; j < kCapPer; ++j) {
        const int i = threadIdx.x + j * 1024;
        if (i < n) {
            const uint32_t tr = bucket[i];
            const int t = static_cast<int>(tr >> 4);
            const float g = gates[static_cast<size_t>(t) * ld + (tr & 15u)];
            const unsigned long long key = (static_cast<unsigned long long>(~__float_as_uint(g)) << 32) | tr;
            const float wt = cap_weight(token_w, t);
            keys[i] = key;
            wts[i] = wt;
            tot += static_cast<unsigned long long>(fixed_weight(wt));
            kmin = min(kmin, key);
            kmax = max(kmax, key);
        }
    }
    for (int off = 16; off >= 1; off >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, off));
        kmax = max(kmax, __shfl_xor_sync(kFull, kmax, off));
    }
    if (threadIdx.x == 0) {
        s_kmin = ~0ull;
        s_kmax = 0ull;
        s_adm = 0ull;
        s_m = 0;
        s_bstar = -1;   // stays -1 only if no bin crosses C: then nothing beyond the load is admitted
        s_excl = 0;
    }
    for (int i = threadIdx.x; i < kCapBins; i += blockDim.x) hist[i] = 0ull;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        atomicMin(&s_kmin, kmin);
        atomicMax(&s_kmax, kmax);
    }
    tot = block_sum_u64(tot, red);   // includes a __syncthreads
    if (n == 0) {
        if (threadIdx.x == 0 && round < 0) w.load[e] = base;
        return;
    }
    if (base + static_cast<long long>(tot) <= C) {
        // everything fits
        for (int i = threadIdx.x; i < n; i += blockDim.x) admit(static_cast<uint32_t>(keys[i] & 0xffffffffull));
        if (threadIdx.x == 0) w.load[e] = base + static_cast<long long>(tot);
        return;
    }
    const unsigned long long k0 = s_kmin, span = s_kmax - s_kmin;
    const int shift = (span >> 10) == 0ull ? 0 : 64 - __clzll(static_cast<long long>(span >> 10));
    auto bin_of = [&](unsigned long long key) { return static_cast<int>((key - k0) >> shift); };
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        atomicAdd(&hist[bin_of(keys[i])], static_cast<unsigned long long>(fixed_weight(wts[i])));
    __syncthreads();
    // exclusive scan of the bins (thread b owns bin b), then the crossing bin
    {
        const int b = threadIdx.x;
        const unsigned long long hv = (b < kCapBins) ? hist[b] : 0ull;
        unsigned long long inc = hv;
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(kFull, inc, off);
            if ((b & 31) >= off) inc += o;
        }
        if ((b & 31) == 31) red[b >> 5] = inc;
        __syncthreads();
        unsigned long long wpre = 0ull;
        for (int i = 0; i < (b >> 5); ++i) wpre += red[i];
        const long long incl = static_cast<long long>(wpre + inc), excl = incl - static_cast<long long>(hv);
        if (b < kCapBins && base + excl <= C && base + incl > C) {
            s_bstar = b;
            s_excl = excl;
        }
    }
    __syncthreads();
    const int bstar = s_bstar;
    const long long excl = s_excl;
    // admit the bins before b*; collect b*'s candidates at the front of keys[]
    unsigned long long mine[kCapPer];
    int nm = 0;
#pragma unroll
    for (int j = 0; j < kCapPer; ++j) {
        const int i = threadIdx.x + j * 1024;
        if (i < n) {
            const unsigned long long key = keys[i];
            const int bb = bin_of(key);
            if (bb < bstar) admit(static_cast<uint32_t>(key & 0xffffffffull));
            else if (bb == bstar) mine[nm++] = key;
        }
    }
    __syncthreads();   // every key is in registers before the front of keys[] is rewritten
    if (nm > 0) {
        const int pos = atomicAdd(&s_m, nm);
        for (int j = 0; j < nm; ++j) keys[pos + j] = mine[j];
    }
    __syncthreads();
    const int m = s_m;
    int P2 = 1;
    while (P2 < m) P2 <<= 1;
    for (int i = m + threadIdx.x; i < P2; i += blockDim.x) keys[i] = ~0ull;
    __syncthreads();
    for (int size = 2; size <= P2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P2 / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long x0 = keys[lo], x1 = keys[hi];
                if ((x0 > x1) == up) {
                    keys[lo] = x1;
                    keys[hi] = x0;
                }
            }
            __syncthreads();
        }
    }
    // running weight through b* in sorted order (m is small: one thread walks it when m <= 64,
    // the weights fetched into shared memory first in one parallel round trip; wts[] is free now)
    if (m <= 64) {
        if (threadIdx.x < m)
            wts[threadIdx.x] = cap_weight(token_w, static_cast<int>((keys[threadIdx.x] & 0xffffffffull) >> 4));
        __syncthreads();
        if (threadIdx.x == 0) {
            long long cum = base + excl;
            unsigned long long adm = 0ull;
            for (int i = 0; i < m; ++i) {
                const uint32_t tr = static_cast<uint32_t>(keys[i] & 0xffffffffull);
                cum += fixed_weight(wts[i]);
                if (cum > C) break;
                admit(tr);
                adm = static_cast<unsigned long long>(cum - base - excl);
            }
            s_adm = adm;
        }
    } else {
        // each thread a contiguous chunk, block scan of the chunk sums
        const int per = (m + blockDim.x - 1) / blockDim.x;
        const int i0 = threadIdx.x * per;
        long long local = 0;
        for (int i = i0; i < min(m, i0 + per); ++i)
            local += fixed_weight(cap_weight(token_w, static_cast<int>((keys[i] & 0xffffffffull) >> 4)));
        unsigned long long inc = static_cast<unsigned long long>(local);
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(kFull, inc, off);
            if ((threadIdx.x & 31) >= off) inc += o;
        }
        __syncthreads();
        if ((threadIdx.x & 31) == 31) red[threadIdx.x >> 5] = inc;
        __syncthreads();
        unsigned long long wpre = 0ull;
        for (int i = 0; i < static_cast<int>(threadIdx.x >> 5); ++i) wpre += red[i];
        long long cum = base + excl + static_cast<long long>(wpre + inc) - local;
        unsigned long long best = 0ull;
        for (int i = i0; i < min(m, i0 + per); ++i) {
            const uint32_t tr = static_cast<uint32_t>(keys[i] & 0xffffffffull);
            cum += fixed_weight(cap_weight(token_w, static_cast<int>(tr >> 4)));
            if (cum > C) break;
            admit(tr);
            best = static_cast<unsigned long long>(cum - base - excl);
        }
        if (best > 0ull) atomicMax(&s_adm, best);
    }
    __syncthreads();
    if (threadIdx.x == 0) w.load[e] = base + excl + static_cast<long long>(s_adm);
}

// Overflow round i: each token offers its lowest-rank pending slot to its
// rank-(k+i) expert.
__global__ void cap_offer_kernel(const int32_t* __restrict__ ids, int ld, int T, int N, int k, int round,
                                 DispatchWs w) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    for (int r = 0; r < k; ++r) {
        if (w.status[static_cast<size_t>(t) * k + r] != kPending) continue;
        const int c = ids[static_cast<size_t>(t) * ld + k + round];
        if (c >= 0 && c < N) {
            const int pos = atomicAdd(&w.cnt2[c], 1);
            if (pos < T)
                w.bucket2[static_cast<size_t>(c) * T + pos] = static_cast<uint32_t>(t) * 16u + static_cast<uint32_t>(r);
        }
        break;
    }
}

// Pending slots are dropped; results are copied out.
__global__ void cap_finalize_kernel(int T, int N, int k, DispatchWs w, uint8_t* slot_status, int64_t* load_q,
                                    int64_t* cap_q, float gamma) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < T * k) {
        if (w.status[i] == kPending) {
            w.status[i] = MOE_SLOT_DROPPED;
            w.wids[i] = -1;
            w.wgates[i] = 0.f;
        } else if (w.status[i] == MOE_SLOT_DROPPED) {
            w.wgates[i] = 0.f;
        }
        if (slot_status) slot_status[i] = w.status[i];
    }
    if (i < N && load_q) load_q[i] = w.load[i];
    if (i == 0 && cap_q) *cap_q = capacity_value(*w.S, k, gamma, N);
}

cudaError_t launch_dispatch(const int32_t* ids, const float* gates, int ld, int T, int N, int k, int R,
                            const float* token_w, float capacity_factor, const int8_t* modality_bias,
                            const float* r_v, int32_t* counts, int32_t* offsets, int32_t* row_token,
                            float* row_gate, int32_t* active, int32_t* out_ids, float* out_gates,
                            int32_t* slot_row, uint8_t* slot_status, int64_t* load_q, int64_t* cap_q, void* ws,
                            moe_dev_status* st, cudaStream_t s) {
    const bool capped = capacity_factor > 0.f;
    DispatchWs w{};
    carve(&w, ws, T, N, k, capped);
    w.bias = modality_bias;
    w.r_v = r_v;
    // an empty batch has no rows: counts, offsets and the active list are zero
    auto clear_empty = [&]() -> cudaError_t {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * N, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (N + 1), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(active, 0, sizeof(int32_t) * (N + 1), s);
        return e;
    };
    if (!capped) {
        if (T == 0) return clear_empty();
        return launch_permute(ids, gates, ld, T, N, k, counts, offsets, row_token, row_gate, active, out_ids,
                              out_gates, slot_row, w.blk_start, st, s);
    }
    cudaError_t err = cudaMemsetAsync(w.S, 0, w.zero_bytes, s);
    if (err != cudaSuccess) return err;
    const int tb = 256;
    if (T > 0) {
        err = launch_pdl(cap_bucket_kernel, dim3((T + 127) / 128), dim3(128), 0, s, ids, gates, ld, T, N, k, token_w,
                         w, st);
        if (err != cudaSuccess) return err;
        size_t P2 = 1;
        while (P2 < static_cast<size_t>(T)) P2 <<= 1;
        const size_t smem = P2 * sizeof(unsigned long long) + static_cast<size_t>(T) * sizeof(float);
        // The kernel's dynamic shared-memory limit is raised once per device
        // to what the largest batch needs and never lowered, so calls of
        // different sizes from several host threads (or a small call before
        // a large captured one) cannot undo each other's setting.
        static std::atomic<bool> attr_set[64] = {};
        int dev = 0;
        err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            err = cudaFuncSetAttribute(cap_admit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kCapAdmitMaxSmem);
            if (err != cudaSuccess) return err;
            attr_set[dev] = true;
        }
        err = launch_pdl(cap_admit_kernel, dim3(N), dim3(1024), smem, s, gates, ld, T, N, k, capacity_factor,
                         token_w, -1, w, st);
        if (err != cudaSuccess) return err;
        for (int i = 0; i + k < R; ++i) {
            err = cudaMemsetAsync(w.cnt2, 0, sizeof(int32_t) * N, s);
            if (err != cudaSuccess) return err;
            err = launch_pdl(cap_offer_kernel, dim3((T + tb - 1) / tb), dim3(tb), 0, s, ids, ld, T, N, k, i, w);
            if (err != cudaSuccess) return err;
            err = launch_pdl(cap_admit_kernel, dim3(N), dim3(1024), smem, s, gates, ld, T, N, k, capacity_factor,
                             token_w, i, w, st);
            if (err != cudaSuccess) return err;
        }
    }
    const int nfin = (T * k > N ? T * k : N);
    err = launch_pdl(cap_finalize_kernel, dim3((nfin + tb - 1) / tb), dim3(tb), 0, s, T, N, k, w, slot_status,
                     load_q, cap_q, capacity_factor);
    if (err != cudaSuccess) return err;
    if (out_ids && T > 0) {
        err = cudaMemcpyAsync(out_ids, w.wids, sizeof(int32_t) * T * k, cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return err;
    }
    if (out_gates && T > 0) {
        err = cudaMemcpyAsync(out_gates, w.wgates, sizeof(float) * T * k, cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return err;
    }
    if (T == 0) return clear_empty();
    return launch_permute(w.wids, w.wgates, k, T, N, k, counts, offsets, row_token, row_gate, active, nullptr,
                          nullptr, slot_row, w.blk_start, st, s);
}

}  // namespace moe
