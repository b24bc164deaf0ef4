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

static inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

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
    static constexpr int X_BYTES = NT * 64 * 2;    // token tile per stage
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int NSTAGE = (NT >= 64) ? 5 : 6;
    static constexpr int ACT_BYTES = NT * BI * 2;  // two 64-column swizzle atoms of NT rows
    static constexpr int NBAR = 2 * NSTAGE + 9;
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + ACT_BYTES + NBAR * 8 + 64;
    static constexpr uint32_t TMEM_COLS = 256;
    static_assert(STAGE % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(4 * NT <= (int)TMEM_COLS, "TMEM columns");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct TcItems {
    int4* items;    // (expert, first row, rows, 0)
    int* n_items;
};

static size_t tc_x_rows(int T, int k) { return static_cast<size_t>(T) * k > 64 ? static_cast<size_t>(T) * k : 64; }

size_t ffn_workspace(int T, int H, int I, int N, int k, int dtype) {
    (void)I;
    if (dtype != MOE_DTYPE_BF16) return 0;
    size_t off = 0;
    off = align_up(off + tc_x_rows(T, k) * H * 2, 256);                                      // X_perm
    off = align_up(off + sizeof(int4) * (static_cast<size_t>(N) + tc_x_rows(T, k) / 16 + 2), 256);  // items
    off = align_up(off + sizeof(int) * 4, 256);                                              // n_items
    return off;
}

static void carve_ffn(void* ws, int T, int H, int N, int k, void** xperm, TcItems* it) {
    char* b = static_cast<char*>(ws);
    size_t off = 0;
    *xperm = b + off;
    off = align_up(off + tc_x_rows(T, k) * H * 2, 256);
    it->items = reinterpret_cast<int4*>(b + off);
    off = align_up(off + sizeof(int4) * (static_cast<size_t>(N) + tc_x_rows(T, k) / 16 + 2), 256);
    it->n_items = reinterpret_cast<int*>(b + off);
}

// ---------------------------------------------------------------------------
// Preparation: gather x rows into expert-sorted order (16-byte vector copies),
// build the work-item list (one item per <= NT-row chunk of each active
// expert) and optionally clear y.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ffn_prep_kernel(const uint4* __restrict__ x, int H, int Mmax,
                                                       const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ row_token,
                                                       const int32_t* __restrict__ active, int N, int NT,
                                                       uint4* __restrict__ xperm, TcItems it, float* y, int T,
                                                       int zero_y) {
    const int M = offsets[N];
    const int vec_per_row = H / 8;  // 8 bf16 per 16 bytes
    const long long total = static_cast<long long>(min(M, Mmax)) * vec_per_row;
    for (long long v = blockIdx.x * 256ll + threadIdx.x; v < total; v += 256ll * gridDim.x) {
        const int row = static_cast<int>(v / vec_per_row), c = static_cast<int>(v % vec_per_row);
        const int tok = row_token[row];
        xperm[v] = x[static_cast<long long>(tok) * vec_per_row + c];
    }
    if (zero_y) {
        const long long ny = static_cast<long long>(T) * H / 4;
        float4* y4 = reinterpret_cast<float4*>(y);
        for (long long v = blockIdx.x * 256ll + threadIdx.x; v < ny; v += 256ll * gridDim.x)
            y4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        // one warp: prefix over active experts of their chunk counts
        const int lane = threadIdx.x;
        const int na = active[0];
        int run = 0;
        for (int base = 0; base < na; base += 32) {
            const int a = base + lane;
            int e = -1, r0 = 0, cnt = 0, ch = 0;
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
            int pos = run + inc - ch;
            for (int c = 0; c < ch; ++c)
                it.items[pos + c] = make_int4(e, r0 + c * NT, min(NT, cnt - c * NT), 0);
            run += __shfl_sync(kFull, inc, 31);
        }
        if (lane == 0) *it.n_items = run;
    }
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

template <int NT>
__global__ void __launch_bounds__(192, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                  const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                  const int4* __restrict__ items, const int* __restrict__ n_items_ptr,
                  const int32_t* __restrict__ row_token, const float* __restrict__ row_gate,
                  float* __restrict__ out, int H, int I, int fuse_combine, moe_dev_status* st) {
    using C = TcCfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = I / C::BI;
    const int n_units = (*n_items_ptr) * S;
    if (static_cast<int>(blockIdx.x) >= n_units) return;

    uint8_t* ring = smem;
    uint8_t* act = smem + C::NSTAGE * C::STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(act + C::ACT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t ring_a = smem_u32(ring), act_a = smem_u32(act);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_G1 = 2 * C::NSTAGE, B_ACTRDY = B_G1 + 1, B_TMEMFREE = B_G1 + 2,
              B_ACTFREE = B_G1 + 3, B_ACC2F = B_G1 + 4, B_ACC2E = B_G1 + 6, B_DRAIN = B_G1 + 8;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_G1), 1);
        mbar_init(bar(B_ACTRDY), 128);
        mbar_init(bar(B_TMEMFREE), 128);
        mbar_init(bar(B_ACTFREE), 1);
        mbar_init(bar(B_ACC2F), 1);
        mbar_init(bar(B_ACC2F + 1), 1);
        mbar_init(bar(B_ACC2E), 128);
        mbar_init(bar(B_ACC2E + 1), 128);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_wg);
        tma_prefetch_desc(&tm_wu);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_x);
    }
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
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, pend = 0, pend_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const int4 it = items[u / S];
                const int s = u % S, e = it.x, row0 = it.y;
                const int wrow = e * I + s * C::BI;
                for (int kt = 0; kt < KT + MT; ++kt) {
                    if (!mbar_wait(bar(B_EMPTY + stage), phase ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring_a + stage * C::STAGE;
                    const uint32_t fb = bar(B_FULL + stage);
                    if (kt < KT) {
                        mbar_arrive_expect_tx(fb, C::STAGE);
                        tma_load_2d(dst, &tm_wg, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BOX, &tm_wu, kt * C::BK, wrow, fb, pol_w);
                        tma_load_2d(dst + C::W_BYTES, &tm_x, kt * C::BK, row0, fb, pol_x);
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
            if (!ok) {
                // let every copy still in flight land before the CTA exits
                for (int i = 0; i < C::NSTAGE; ++i)
                    if (pend >> i & 1u) mbar_drain(bar(B_FULL + i), pend_par >> i & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t idesc = idesc_bf16_f32(128, NT);
            int stage = 0, j = 0;
            uint32_t phase = 0, n2 = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++j) {
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
                    const uint32_t b = n2 & 1u, use = n2 >> 1;
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
        // ---------------- epilogue: warps 2..5 ----------------
        const int q = warp & 3;               // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;        // row within the 128-row tile
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        int j = 0;
        uint32_t n2 = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
            const int4 it = items[u / S];
            const int s = u % S, row0 = it.y, nrows = it.z;
            // every lane polls; the warp proceeds only if all lanes saw the phase complete
            bool okw = mbar_wait(bar(B_G1), j & 1, abort_flag, st, kSiteEpiG1Done);
            if (!__all_sync(kFull, okw)) break;
            okw = mbar_wait(bar(B_ACTFREE), (j & 1) ^ 1, abort_flag, st, kSiteEpiActFree);
            if (!__all_sync(kFull, okw)) break;
            tc_fence_after();
            // SwiGLU of this thread's I row for every token of the chunk -> bf16 B operand of GEMM2
            const int c = row >> 6, ci = row & 63;
            const uint32_t col_base = act_a + c * (NT * 128);
#pragma unroll
            for (int c0 = 0; c0 < NT / 16; ++c0) {
                uint32_t g[16], v[16];
                tmem_ld16(t_gate + lane_off + c0 * 16, g);
                tmem_ld16(t_up + lane_off + c0 * 16, v);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int t = c0 * 16 + jj;
                    const float a = (t < nrows) ? silu_mul(__uint_as_float(g[jj]), __uint_as_float(v[jj])) : 0.f;
                    const __nv_bfloat16 hb = __float2bfloat16_rn(a);
                    const uint32_t addr =
                        col_base + t * 128 + ((((ci >> 3) ^ (t & 7)) << 4) | ((ci & 7) << 1));
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<const uint16_t*>(&hb))
                                 : "memory");
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_TMEMFREE));
            fence_proxy_async_smem();
            mbar_arrive(bar(B_ACTRDY));
            // down projection tiles: add gate * E_e(x) into y
            bool ok = true;
            for (int m = 0; m < H / C::BH; ++m, ++n2) {
                const uint32_t b = n2 & 1u, use = n2 >> 1;
                const bool okw2 = mbar_wait(bar(B_ACC2F + b), use & 1u, abort_flag, st, kSiteEpiAcc2Full);
                if (!__all_sync(kFull, okw2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int h = m * C::BH + row;
#pragma unroll
                for (int c0 = 0; c0 < NT / 16; ++c0) {
                    uint32_t v[16];
                    tmem_ld16(t_acc2 + b * NT + lane_off + c0 * 16, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int t = c0 * 16 + jj;
                        if (t < nrows) {
                            const float val = __uint_as_float(v[jj]);
                            if (fuse_combine) {
                                const int tok = row_token[row0 + t];
                                const float gt = row_gate[row0 + t];
                                atomicAdd(out + static_cast<size_t>(tok) * H + h, gt * val);
                            } else {
                                atomicAdd(out + static_cast<size_t>(row0 + t) * H + h, val);
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(B_ACC2E + b));
            }
            if (!ok) break;
            (void)s;
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

template <int NT>
static cudaError_t run_tc(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I, int N,
                          int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                          const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                          cudaStream_t s) {
    using C = TcCfg<NT>;
    void* xperm = nullptr;
    TcItems it{};
    carve_ffn(ws, T, H, N, k, &xperm, &it);
    const size_t xrows = tc_x_rows(T, k);
    const int Mmax = T * k;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    const int zero_y = (fuse && (flags & MOE_FFN_ZERO_Y)) ? 1 : 0;
    {
        const long long work = static_cast<long long>(Mmax) * (H / 8);
        int grid = static_cast<int>((work + 255) / 256);
        grid = grid < 1 ? 1 : (grid > 1024 ? 1024 : grid);
        ffn_prep_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(x), H, Mmax, offsets, row_token, active, N,
                                             NT, static_cast<uint4*>(xperm), it, out, T, zero_y);
    }
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x;
    if (!make_tmap(&tm_wg, wg, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wu, wu, H, static_cast<uint64_t>(N) * I, 64, 128) ||
        !make_tmap(&tm_wd, wd, I, static_cast<uint64_t>(N) * H, 64, 128) ||
        !make_tmap(&tm_x, xperm, H, xrows, 64, NT))
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
    const long long max_items = (N < Mmax ? N : Mmax) + (Mmax + NT - 1) / NT;
    long long max_units = max_items * (I / C::BI);
    int grid = sm_count();
    if (max_units < grid) grid = static_cast<int>(max_units > 0 ? max_units : 1);
    ffn_tc_kernel<NT><<<grid, 192, C::SMEM, s>>>(tm_wg, tm_wu, tm_wd, tm_x, it.items, it.n_items, row_token,
                                                 row_gate, out, H, I, fuse ? 1 : 0, st);
    return cudaGetLastError();
}

cudaError_t launch_ffn_bf16(const void* x, const void* wg, const void* wu, const void* wd, int T, int H, int I,
                            int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                            const int32_t* active, uint32_t flags, float* out, void* ws, moe_dev_status* st,
                            cudaStream_t s) {
    if (T <= 16) return run_tc<16>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, ws, st, s);
    if (T <= 32) return run_tc<32>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, ws, st, s);
    return run_tc<64>(x, wg, wu, wd, T, H, I, N, k, offsets, row_token, row_gate, active, flags, out, ws, st, s);
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
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += 256ll * gridDim.x) p[i] = 0.f;
}

cudaError_t launch_ffn_f32(const float* x, const float* wg, const float* wu, const float* wd, int T, int H, int I,
                           int N, int k, const int32_t* offsets, const int32_t* row_token, const float* row_gate,
                           const int32_t* active, uint32_t flags, float* out, moe_dev_status* st, cudaStream_t s) {
    (void)active;
    (void)st;
    const bool fuse = (flags & MOE_FFN_FUSE_COMBINE) != 0;
    if (fuse && (flags & MOE_FFN_ZERO_Y)) {
        const long long n = static_cast<long long>(T) * H;
        int grid = static_cast<int>((n + 255) / 256);
        grid = grid < 1 ? 1 : (grid > 1024 ? 1024 : grid);
        zero_kernel<<<grid, 256, 0, s>>>(out, n);
    }
    const int Mmax = T * k;
    if (Mmax == 0) return cudaGetLastError();
    const size_t smem = sizeof(float) * static_cast<size_t>(H + I);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(ffn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    ffn_f32_kernel<<<Mmax, 256, smem, s>>>(x, wg, wu, wd, H, I, N, offsets, row_token, row_gate, fuse ? 1 : 0, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Deterministic combine: y[t] = sum over slots (in slot order) of gate * row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ rows_out,
                                                      const int32_t* __restrict__ slot_row,
                                                      const float* __restrict__ slot_gate, int T, int H, int k,
                                                      float* __restrict__ y) {
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
    combine_kernel<<<grid, 256, 0, s>>>(rows_out, slot_row, slot_gate, T, H, k, y);
    return cudaGetLastError();
}

}  // namespace moe
