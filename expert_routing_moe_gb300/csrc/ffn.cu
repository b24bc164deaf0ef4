// ffn.cu -- grouped SwiGLU expert FFN with the weighted combine fused in.
//
// E_j(x) = W_down_j (silu(W_gate_j x) * (W_up_j x)) and
// y(x) = sum_j G(x)_j E_j(x): "MACS: Modality-Aware Capacity Scaling for
// Efficient Multimodal MoE Inference", sec. 3.1, Eq. (1).  Only the experts
// that received rows are visited, so the bytes moved per layer are the
// active experts' weights (the decode bottleneck the SERE article measures in
// sec. 1.2 / 2.2).
//
// bf16 path (tensor cores): a persistent kernel, one CTA per SM, walks work
// units (expert e, token chunk of <= NT rows, 128-row slice of I).  For a
// unit it streams W_gate/W_up[e][slice][:] and W_down[e][:][slice] once
// through a TMA ring in shared memory and runs two tcgen05 GEMMs with the
// weights as the 128-row MMA operand and the tokens as the N operand:
//   GEMM1  D_g, D_u [128 x NT] = W_{gate,up}[slice] . X_chunk^T    (K = H)
//   SwiGLU A = silu(D_g) * D_u  -> bf16 in shared memory            (epilogue)
//   GEMM2  D_y [128 x NT] = W_down[h-tile][slice] . A^T            (K = 128)
// and adds gate * D_y into y with coalesced fp32 reductions.  Warp roles:
// warp 0 TMA producer, warp 1 MMA issuer + TMEM owner, warps 2-5 epilogue.
// fp32 path: a CUDA-core kernel, one CTA per row.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace moe {


// ---------------------------------------------------------------------------
// Tile configuration of the tensor-core kernel.
// ---------------------------------------------------------------------------
template <int NT>
struct TcCfg {
    static constexpr int BI = 128;                 // slice of I per unit (GEMM1 M)
    static constexpr int BK = 64;                  // K tile: 64 bf16 = one 128-byte swizzle row
    static constexpr int BH = 128;                 // H tile of GEMM2 (GEMM2 M)
    static constexpr int W_BOX = 128 * 64 * 2;     // one 128x64 bf16 box = 16 KiB
    static constexpr int W_BYTES = 2 * W_BOX;      // two boxes per stage
    static constexpr int X_BYTES = NT * 64 * 2;    // token tile per stage (NT gathered rows)
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int NSTAGE = (NT <= 16) ? 6 : 5;
    static constexpr int ACT_BYTES = NT * BI * 2;  // two 64-column swizzle atoms of NT rows
    static constexpr int NACC2 = (NT <= 32) ? 4 : 2;
    static constexpr int EPI_WARPS = 8;            // two warps per TMEM lane quadrant
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int CW = NT / 2;              // token columns per epilogue warp
    static constexpr int NBAR = 2 * NSTAGE + 5 + 2 * NACC2;
    static constexpr int TABLE_INTS = 4 * MOE_MAX_EXPERTS + 4;
    static constexpr int SMEM =
        1024 + NSTAGE * STAGE + ACT_BYTES + NBAR * 8 + 16 + 64 * 4 + TABLE_INTS * 4 + EPI_WARPS * 32 * 8;
    static constexpr uint32_t TMEM_COLS = 256;
    static_assert(STAGE % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert((2 + NACC2) * NT <= (int)TMEM_COLS, "TMEM columns");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(CW == 8 || CW == 16 || CW == 32, "epilogue column split");
};

size_t ffn_workspace(int T, int H, int I, int N, int k, int dtype) {
    (void)T; (void)H; (void)I; (void)N; (void)k; (void)dtype;
    return 0;  // the tensor-core path reads token rows straight from x
}

// Work units: for every active expert a, ceil(rows/NT) token chunks, each
// split into I/128 slices.  The table (built once per CTA in shared memory)
// holds, per active expert, its id, first row, row count and first chunk.
struct UnitTable {
    int* e;      // [na]
    int* row;    // [na]
    int* cnt;    // [na]
    int* pre;    // [na + 1]: exclusive prefix of chunk counts
    int na;
};

__device__ __forceinline__ void unit_info(const UnitTable& tb, int u, int S, int NT, int& e, int& s, int& row0,
                                          int& nrows) {
    const int item = u / S;
    s = u - item * S;
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

// ---------------------------------------------------------------------------
// The tensor-core kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[CW]) {
    if constexpr (CW == 8) {
        tmem_ld8(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < CW / 16; ++c) {
            uint32_t w[16];
            tmem_ld16(taddr + c * 16, w);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[c * 16 + j] = w[j];
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(TcCfg<NT>::THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                  const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ active,
                  const int32_t* __restrict__ row_token, const float* __restrict__ row_gate,
                  float* __restrict__ out, int H, int I, int N, int fuse_combine, moe_dev_status* st) {
    using C = TcCfg<NT>;
    constexpr int CW = C::CW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* act = smem + C::NSTAGE * C::STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(act + C::ACT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_units = reinterpret_cast<int*>(tmem_slot + 2);
    int* ptok = reinterpret_cast<int*>(tmem_slot + 4);           // [64] token rows of the producer's unit
    int* table = ptok + 64;
    int* etok_all = table + C::TABLE_INTS;                           // [EPI_WARPS][32] tokens of each epilogue warp
    float* egt_all = reinterpret_cast<float*>(etok_all + C::EPI_WARPS * 32);  // [EPI_WARPS][32] their gates
    UnitTable tb{table, table + MOE_MAX_EXPERTS, table + 2 * MOE_MAX_EXPERTS, table + 3 * MOE_MAX_EXPERTS, 0};

    const uint32_t ring_a = smem_u32(ring), act_a = smem_u32(act);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_G1 = 2 * C::NSTAGE, B_ACTRDY = B_G1 + 1, B_TMEMFREE = B_G1 + 2,
              B_ACTFREE = B_G1 + 3, B_DRAIN = B_G1 + 4, B_ACC2F = B_G1 + 5, B_ACC2E = B_ACC2F + C::NACC2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_G1), 1);
        mbar_init(bar(B_ACTRDY), C::EPI_THREADS);
        mbar_init(bar(B_TMEMFREE), C::EPI_THREADS);
        mbar_init(bar(B_ACTFREE), 1);
        mbar_init(bar(B_DRAIN), 1);
        for (int b = 0; b < C::NACC2; ++b) {
            mbar_init(bar(B_ACC2F + b), 1);
            mbar_init(bar(B_ACC2E + b), C::EPI_THREADS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_wg);
        tma_prefetch_desc(&tm_wu);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_x);
    }
    // everything above is private to this CTA; the dispatch outputs and y are read below
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        // work-unit table: prefix over active experts of their chunk counts
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
            s_units[0] = na;
            s_units[1] = run * (I / C::BI);
        }
    }
    __syncthreads();
    tb.na = s_units[0];
    const int n_units = s_units[1];
    const int S = I / C::BI;
    if (static_cast<int>(blockIdx.x) >= n_units) return;
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_gate = tmem, t_up = tmem + NT, t_acc2 = tmem + 2 * NT;
    const int KT = H / C::BK, MT = H / C::BH;

    if (warp == 0) {
        // ---------------- TMA producer (lane 0 issues; the warp loads token lists) ----------------
        const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, pend = 0, pend_par = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            int e, s, row0, nrows;
            unit_info(tb, u, S, NT, e, s, row0, nrows);
            // rows past the chunk repeat its first token; their columns are never used
            for (int t = lane; t < NT; t += 32) ptok[t] = row_token[row0 + (t < nrows ? t : 0)];
            __syncwarp();
            if (lane == 0) {
                const int wrow = e * I + s * C::BI;
                const int n_g4 = (nrows + 3) / 4;
                for (int kt = 0; kt < KT + MT; ++kt) {
                    if (!mbar_wait(bar(B_EMPTY + stage), phase ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring_a + stage * C::STAGE;
                    const uint32_t fb = bar(B_FULL + stage);
                    if (kt < KT) {
                        // only the gathers that hold real rows; the MMA's N covers them, rows past
                        // nrows in the last 16-row group belong to columns that are never used
                        mbar_arrive_expect_tx(fb, C::W_BYTES + n_g4 * 512);
                        tma_load_2d(dst, &tm_wg, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wu, kt * C::BK, wrow, fb, pol_w);
                        for (int g = 0; g < n_g4; ++g)
                            tma_gather4(dst + C::W_BYTES + g * 512, &tm_x, kt * C::BK, ptok[4 * g], ptok[4 * g + 1],
                                        ptok[4 * g + 2], ptok[4 * g + 3], fb, pol_x);
                    } else {
                        const int m = kt - KT;
                        mbar_arrive_expect_tx(fb, C::W_BYTES);
                        tma_load_2d(dst, &tm_wd, s * C::BI, e * H + m * C::BH, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wd, s * C::BI + 64, e * H + m * C::BH, fb, pol_w);
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
            int stage = 0, j = 0;
            uint32_t phase = 0, n2 = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++j) {
                // the MMA's N is the unit's row count rounded up to 16
                int ue, us, urow0, unrows;
                unit_info(tb, u, S, NT, ue, us, urow0, unrows);
                const int n_eff = min(NT, max(16, (unrows + 15) & ~15));
                const uint32_t idesc = idesc_bf16_f32(128, n_eff);
                if (!mbar_wait(bar(B_TMEMFREE), (j & 1) ^ 1, abort_flag, st, kSiteMmaTmemFree)) break;
                tc_fence_after();
                for (int kt = 0; kt < KT && ok; ++kt) {
                    if (!mbar_wait(bar(B_FULL + stage), phase, abort_flag, st, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring_a + stage * C::STAGE;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk) {
                        const uint64_t dg = sw128_desc(a + kk * 32);
                        const uint64_t du = sw128_desc(a + C::W_BOX + kk * 32);
                        const uint64_t dx = sw128_desc(a + C::W_BYTES + kk * 32);
                        const uint32_t acc = (kt | kk) != 0;
                        tc_mma_bf16(t_gate, dg, dx, idesc, acc);
                        tc_mma_bf16(t_up, du, dx, idesc, acc);
                    }
                    tc_commit(bar(B_EMPTY + stage));
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar(B_G1));
                if (!mbar_wait(bar(B_ACTRDY), j & 1, abort_flag, st, kSiteMmaActReady)) break;
                tc_fence_after();
                for (int m = 0; m < MT; ++m, ++n2) {
                    if (!mbar_wait(bar(B_FULL + stage), phase, abort_flag, st, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b = n2 % C::NACC2, use = n2 / C::NACC2;
                    if (!mbar_wait(bar(B_ACC2E + b), (use & 1u) ^ 1u, abort_flag, st, kSiteMmaAcc2Empty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring_a + stage * C::STAGE;
#pragma unroll
                    for (int kk = 0; kk < C::BI / 16; ++kk) {
                        const uint64_t dw = sw128_desc(a + (kk >> 2) * C::W_BOX + (kk & 3) * 32);
                        const uint64_t da = sw128_desc(act_a + (kk >> 2) * (NT * 128) + (kk & 3) * 32);
                        tc_mma_bf16(t_acc2 + b * NT, dw, da, idesc, kk != 0);
                    }
                    tc_commit(bar(B_EMPTY + stage));
                    tc_commit(bar(B_ACC2F + b));
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar(B_ACTFREE));
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
        const int row = q * 32 + lane;                 // row within the 128-row tile
        const int c_lo = half * CW;                    // first token column of this warp
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int c = row >> 6, ci = row & 63;
        int j = 0;
        uint32_t n2 = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
            int e, s, row0, nrows;
            unit_info(tb, u, S, NT, e, s, row0, nrows);
            // every lane polls; the warp proceeds only if all lanes saw the phase complete
            bool okw = mbar_wait(bar(B_G1), j & 1, abort_flag, st, kSiteEpiG1Done);
            if (!__all_sync(kFull, okw)) break;
            okw = mbar_wait(bar(B_ACTFREE), (j & 1) ^ 1, abort_flag, st, kSiteEpiActFree);
            if (!__all_sync(kFull, okw)) break;
            tc_fence_after();
            {
                // SwiGLU of this thread's I row for its token columns -> bf16 B operand of GEMM2,
                // eight columns at a time
                const uint32_t col_base = act_a + c * (NT * 128);
#pragma unroll
                for (int c8 = 0; c8 < CW / 8; ++c8) {
                    uint32_t g[8], v[8];
                    if (c_lo + c8 * 8 < nrows) {   // warp-uniform
                        tmem_ld8(t_gate + lane_off + c_lo + c8 * 8, g);
                        tmem_ld8(t_up + lane_off + c_lo + c8 * 8, v);
                        tmem_ld_wait();
                    }
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int t = c_lo + c8 * 8 + jj;
                        const float a =
                            (t < nrows) ? silu_mul(__uint_as_float(g[jj]), __uint_as_float(v[jj])) : 0.f;
                        const __nv_bfloat16 hb = __float2bfloat16_rn(a);
                        const uint32_t addr = col_base + t * 128 + ((((ci >> 3) ^ (t & 7)) << 4) | ((ci & 7) << 1));
                        asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                                     "h"(*reinterpret_cast<const uint16_t*>(&hb))
                                     : "memory");
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_TMEMFREE));
            fence_proxy_async_smem();
            mbar_arrive(bar(B_ACTRDY));
            // token and gate of each of this warp's columns, for the reductions below
            int* etok = etok_all + (warp - 2) * 32;
            float* egt = egt_all + (warp - 2) * 32;
            if (lane < CW) {
                const int t = c_lo + lane;
                etok[lane] = (t < nrows) ? row_token[row0 + t] : 0;
                egt[lane] = (t < nrows) ? row_gate[row0 + t] : 0.f;
            }
            __syncwarp();
            // down-projection tiles: add gate * E_e(x) into y
            bool ok = true;
            for (int m = 0; m < H / C::BH; ++m, ++n2) {
                const uint32_t b = n2 % C::NACC2, use = n2 / C::NACC2;
                const bool okw2 = mbar_wait(bar(B_ACC2F + b), use & 1u, abort_flag, st, kSiteEpiAcc2Full);
                if (!__all_sync(kFull, okw2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // read the accumulator in chunks of up to 16 columns; it is released right
                // after the last read, before the last chunk's reductions
                constexpr int CH = CW < 16 ? CW : 16;
                const int h = m * C::BH + row;
#pragma unroll
                for (int c16 = 0; c16 < CW / CH; ++c16) {
                    const bool any = c_lo + c16 * CH < nrows;   // warp-uniform
                    uint32_t v[CH];
                    if (any) {
                        if constexpr (CH == 8) {
                            tmem_ld8(t_acc2 + b * NT + lane_off + c_lo, v);
                        } else {
                            tmem_ld16(t_acc2 + b * NT + lane_off + c_lo + c16 * CH, v);
                        }
                        tmem_ld_wait();
                    }
                    if (c16 == CW / CH - 1) {
                        tc_fence_before();
                        mbar_arrive(bar(B_ACC2E + b));
                    }
                    if (!any) continue;
#pragma unroll
                    for (int jj = 0; jj < CH; ++jj) {
                        const int t = c_lo + c16 * CH + jj;
                        const int js = c16 * CH + jj;   // index into this warp's token slice
                        if (t < nrows) {
                            if (fuse_combine)
                                atomicAdd(out + static_cast<size_t>(etok[js]) * H + h, egt[js] * __uint_as_float(v[jj]));
                            else
                                atomicAdd(out + static_cast<size_t>(row0 + t) * H + h, __uint_as_float(v[jj]));
                        }
                    }
                }
            }
            __syncwarp();   // the warp's token slice is rewritten for the next unit
            if (!ok) break;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side of the tensor-core path.
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// boxes of box_inner x box_outer with the 128-byte swizzle.
static bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

__global__ void zero_kernel(float* p, long long n);

static cudaError_t launch_zero(float* p, long long n, cudaStream_t s) {
    int grid = static_cast<int>((n / 4 + 255) / 256);
    grid = grid < 1 ? 1 : (grid > 1024 ? 1024 : grid);
    return launch_pdl(zero_kernel, dim3(grid), dim3(256), 0, s, p, n);
}

template <int NT>
static cudaError_t run_tc(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I, int N,
                          int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                          const int32_t* active, uint32_t flags, float* out, moe_dev_status* st, cudaStream_t s) {
    using C = TcCfg<NT>;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    if (fuse && (flags & MOE_FFN_ZERO_Y)) {
        cudaError_t e = launch_zero(out, static_cast<long long>(T) * H, s);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x;
    if (!make_tmap(&tm_wg, wg, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wu, wu, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wd, wd, I, static_cast<uint64_t>(N) * H, 64, 128) ||
        !make_tmap(&tm_x, x, H, static_cast<uint64_t>(T), 64, 1))
        return cudaErrorInvalidValue;
    // the attribute is set once per device, on the first (uncaptured) call
    static bool attr_set[64] = {};
    int devi = 0;
    cudaGetDevice(&devi);
    if (devi < 0 || devi >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[devi]) {
        cudaError_t ae = cudaFuncSetAttribute(ffn_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (ae != cudaSuccess) return ae;
        attr_set[devi] = true;
    }
    const int Mmax = T * k;
    const long long max_items = (N < Mmax ? N : Mmax) + (Mmax + NT - 1) / NT;
    const long long max_units = max_items * (I / C::BI);
    int grid = sm_count();
    if (max_units < grid) grid = static_cast<int>(max_units > 0 ? max_units : 1);
    return launch_pdl(ffn_tc_kernel<NT>, dim3(grid), dim3(C::THREADS), C::SMEM, s, tm_wg, tm_wu, tm_wd, tm_x, offsets,
                      active, row_token, row_gate, out, H, I, N, fuse ? 1 : 0, st);
}

cudaError_t launch_ffn_bf16(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                            int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                            const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                            cudaStream_t s) {
    (void)ws;
    if (T <= 16) return run_tc<16>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, st, s);
    if (T <= 32) return run_tc<32>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, st, s);
    return run_tc<64>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, st, s);
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

__global__ void zero_kernel(float* p, long long n) {
    pdl_wait();
    pdl_trigger();
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
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(ffn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
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
