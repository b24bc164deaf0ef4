// permute.cuh -- pieces of the expert-sorted permutation (rows ordered by
// (expert asc, token asc)), shared by the dispatch kernels and the fused
// decode layer kernel.  A row's position is its expert's start plus the
// number of earlier tokens holding that expert, counted with a per-expert
// presence bitmap over a block of up to 1024 tokens and population counts,
// so the order is deterministic without a sort.  "MACS" sec. 3.1 (the token
// sets I_j of Eq. (2)).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kBlk = 1024;          // tokens per permutation block (one per thread)
constexpr int kWordsPerBlk = kBlk / 32;

// ---------------------------------------------------------------------------
// Permutation
// ---------------------------------------------------------------------------
// Marks, for the 1024-token block `b`, bit (t mod 1024) of expert e's bitmap
// for every slot of token t holding e.
// nw = 32-bit words per expert (tokens of the block / 32, rounded up).
__device__ __forceinline__ void presence_bits(const int32_t* __restrict__ ids, int ld, int T, int N, int k, int b, int nw,
                              uint32_t* bits, moe_dev_status* st) {
    for (int i = threadIdx.x; i < N * nw; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    const int t = b * kBlk + threadIdx.x;
    if (t < T && threadIdx.x < nw * 32) {
        for (int r = 0; r < k; ++r) {
            const int e = ids[static_cast<size_t>(t) * ld + r];
            if (e >= N) report(st, MOE_DEV_BAD_INDEX, e);
            if (e >= 0 && e < N) atomicOr(&bits[e * nw + (threadIdx.x >> 5)], 1u << (threadIdx.x & 31));
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int block_count(const uint32_t* bits, int e, int nw) {
    int c = 0;
    for (int w = 0; w < nw; ++w) c += __popc(bits[e * nw + w]);
    return c;
}

// Writes the rows of block b given the absolute start row of each expert in
// this block (start[e]).
__device__ __forceinline__ void write_rows(const int32_t* __restrict__ ids, const float* __restrict__ gates, int ld, int T, int N,
                           int k, int b, int nw, const uint32_t* bits, const int32_t* start,
                           int32_t* __restrict__ row_token,
                           float* __restrict__ row_gate, int32_t* __restrict__ out_ids,
                           float* __restrict__ out_gates, int32_t* __restrict__ slot_row) {
    const int t = b * kBlk + threadIdx.x;
    if (t >= T || threadIdx.x >= nw * 32) return;
    const int w0 = threadIdx.x >> 5;
    const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
    for (int r = 0; r < k; ++r) {
        const size_t si = static_cast<size_t>(t) * ld + r;
        const size_t so = static_cast<size_t>(t) * k + r;
        const int e = ids[si];
        const float g = gates[si];
        int row = -1;
        if (e >= 0 && e < N) {
            int c = 0;
            for (int w = 0; w < w0; ++w) c += __popc(bits[e * nw + w]);
            c += __popc(bits[e * nw + w0] & below);
            row = start[e] + c;
            row_token[row] = t;
            row_gate[row] = g;
        }
        if (slot_row) slot_row[so] = row;
        if (out_ids) out_ids[so] = (row >= 0) ? e : -1;
        if (out_gates) out_gates[so] = (row >= 0) ? g : 0.f;
    }
}

// Exclusive scan of counts over experts; fills offsets and the active list.
// Runs in one CTA with blockDim >= N.
__device__ __forceinline__ void scan_experts(const int* cnt_total, int N, int32_t* counts, int32_t* offsets, int32_t* active,
                             int* s_off) {
    // N <= 256: a simple two-level scan by the first warp
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int run = 0, arun = 0;
        for (int base = 0; base < N; base += 32) {
            const int e = base + lane;
            const int c = (e < N) ? cnt_total[e] : 0;
            const int a = (c > 0) ? 1 : 0;
            int inc = c, ainc = a;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFull, inc, off);
                const int av = __shfl_up_sync(kFull, ainc, off);
                if (lane >= off) {
                    inc += v;
                    ainc += av;
                }
            }
            if (e < N) {
                s_off[e] = run + inc - c;
                counts[e] = c;
                offsets[e] = run + inc - c;
                if (a) active[1 + arun + ainc - 1] = e;
            }
            run += __shfl_sync(kFull, inc, 31);
            arun += __shfl_sync(kFull, ainc, 31);
        }
        if (lane == 0) {
            offsets[N] = run;
            active[0] = arun;
        }
    }
}

}  // namespace moe
