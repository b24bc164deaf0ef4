// router.cu -- router GEMM, fp32 softmax gate + top-R ranking, and the SERE
// batch reroute fused into the ranking kernel.
//
// Router and gate: "MACS: Modality-Aware Capacity Scaling for Efficient
// Multimodal MoE Inference", sec. 3.1, Eq. (1).
// SERE: Xiaohongshu multi-image QA inference article, sec. 4.1 (primary
// union as the shared candidate set, most-similar primary above rho) and
// sec. 4.2 (one fused operator, protection of source experts only).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "routing.cuh"
#include "tmap.h"

namespace moe {

// ---------------------------------------------------------------------------
// Router GEMM, small batches: router_tile (routing.cuh) with two experts per
// 256-thread CTA, grid (ceil(N/2), ceil(T/4)).
// ---------------------------------------------------------------------------
template <typename XT>
__global__ void __launch_bounds__(256) router_warp_kernel(const XT* __restrict__ x, const float* __restrict__ w,
                                                          int T, int H, int N, float* __restrict__ logits) {
    __shared__ float part[8][4];
    pdl_wait();
    pdl_trigger();
    router_tile<XT, 2>(x, w, T, H, N, blockIdx.x * 2, blockIdx.y * 4, logits, part);
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
    pdl_wait();
    pdl_trigger();
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


// ---------------------------------------------------------------------------
// Router GEMM on the tensor cores, large batches of bf16 tokens.
//
// W_r is fp32.  Each element is split exactly into three bf16 parts,
// w = hi + mid + lo (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid);
// both differences are exact in fp32 and lo carries the last bits to within
// 2^-27 |w|), so every bf16 x bf16 product is exact and the tcgen05 MMA sums
// x.w over the three planes with fp32 accumulation.  CTA = 128 tokens x 64
// experts.  Per 64-wide K chunk: warp 0 brings the x tile (TMA, 128-byte
// swizzle) and the fp32 W chunk (TMA, unswizzled) into a 3-stage ring; warps
// 2-5 split W into three swizzled bf16 planes; warp 1 issues 3 x 4 MMAs of
// 128 x 64 x 16 into a 64-column TMEM accumulator.  Warps 2-5 then store the
// logits.  Every wait is bounded.
// ---------------------------------------------------------------------------
constexpr int kRouterTcMinT = 256;   // larger batches use the tensor-core router

struct RtCfg {
    static constexpr int BM = 128, BN = 64, BK = 64;
    static constexpr int X_BYTES = BM * BK * 2;      // 16 KiB, bf16 tokens
    static constexpr int PLANE = BN * BK * 2;        // 8 KiB, one bf16 part of W
    static constexpr int W32_BYTES = BN * BK * 4;    // 16 KiB, the fp32 W chunk
    static constexpr int OFF_PLANES = X_BYTES;
    static constexpr int OFF_W32 = X_BYTES + 3 * PLANE;
    static constexpr int STAGE = X_BYTES + 3 * PLANE + W32_BYTES;   // 56 KiB
    static constexpr int NSTAGE = 3;
    static constexpr int THREADS = 192;
    static constexpr int CONV_THREADS = 128;
    static constexpr int NBAR = 3 * NSTAGE + 2;
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + NBAR * 8 + 16;
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
};

__global__ void __launch_bounds__(RtCfg::THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int T,
                     int H, int N, float* __restrict__ logits, moe_dev_status* st) {
    using C = RtCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::NSTAGE * C::STAGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t ring_a = smem_u32(smem);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_CONV = C::NSTAGE, B_EMPTY = 2 * C::NSTAGE, B_ACC = 3 * C::NSTAGE, B_DRAIN = B_ACC + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * C::BM, n0 = blockIdx.y * C::BN;
    const int KT = H / C::BK;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_CONV + i), C::CONV_THREADS);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_ACC), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::BN);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            uint32_t pend = 0, pend_par = 0;
            bool ok = true;
            for (int c = 0; c < KT; ++c) {
                const int s = c % C::NSTAGE;
                const uint32_t ph = (c / C::NSTAGE) & 1;
                if (!mbar_wait(bar(B_EMPTY + s), ph ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = ring_a + s * C::STAGE;
                mbar_arrive_expect_tx(bar(B_FULL + s), C::X_BYTES + C::W32_BYTES);
                tma_load_2d(dst, &tm_x, c * C::BK, t0, bar(B_FULL + s), pol);
                tma_load_2d(dst + C::OFF_W32, &tm_w, c * C::BK, n0, bar(B_FULL + s), pol);
                pend |= 1u << s;
                pend_par = (pend_par & ~(1u << s)) | (ph << s);
            }
            if (!ok)
                for (int i = 0; i < C::NSTAGE; ++i)
                    if (pend >> i & 1u) mbar_drain(bar(B_FULL + i), pend_par >> i & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(C::BM, C::BN);
            bool ok = true;
            for (int c = 0; c < KT && ok; ++c) {
                const int s = c % C::NSTAGE;
                if (!mbar_wait(bar(B_CONV + s), (c / C::NSTAGE) & 1, abort_flag, st, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = ring_a + s * C::STAGE;
#pragma unroll
                for (int p = 0; p < 3; ++p)
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc_mma_bf16(tmem, sw128_desc(a + kk * 32), sw128_desc(a + C::OFF_PLANES + p * C::PLANE + kk * 32),
                                    idesc, (c | p | kk) != 0);
                tc_commit(bar(B_EMPTY + s));
            }
            if (ok) tc_commit(bar(B_ACC));
            tc_commit(bar(B_DRAIN));
            mbar_drain(bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        // ---- split W into three bf16 planes (swizzled K-major), then the epilogue ----
        const int ct = threadIdx.x - 64;           // 0..127
        const int r = ct >> 1, kh = ct & 1;        // W row (expert) and which half of the 64 k
        bool ok = true;
        for (int c = 0; c < KT; ++c) {
            const int s = c % C::NSTAGE;
            ok = __all_sync(kFull, mbar_wait(bar(B_FULL + s), (c / C::NSTAGE) & 1, abort_flag, st, kSiteEpiG1Done));
            if (!ok) break;
            uint8_t* stage = smem + s * C::STAGE;
            const float* wrow = reinterpret_cast<const float*>(stage + C::OFF_W32) + r * C::BK + kh * 32;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = (jj + r) & 3;            // rotated so that neighbouring rows use other banks
                const float4 a = reinterpret_cast<const float4*>(wrow)[2 * j];
                const float4 b = reinterpret_cast<const float4*>(wrow)[2 * j + 1];
                const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                uint32_t ph[4], pm[4], pl[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * q]), h1 = __float2bfloat16_rn(v[2 * q + 1]);
                    const float r0 = __fsub_rn(v[2 * q], __bfloat162float(h0));
                    const float r1 = __fsub_rn(v[2 * q + 1], __bfloat162float(h1));
                    __nv_bfloat16 m0 = __float2bfloat16_rn(r0), m1 = __float2bfloat16_rn(r1);
                    __nv_bfloat16 l0 = __float2bfloat16_rn(__fsub_rn(r0, __bfloat162float(m0)));
                    __nv_bfloat16 l1 = __float2bfloat16_rn(__fsub_rn(r1, __bfloat162float(m1)));
                    ph[q] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
                    pm[q] = static_cast<uint32_t>(__bfloat16_as_ushort(m0)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(m1)) << 16);
                    pl[q] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
                }
                // 16-byte chunk (kh*4 + j) of row r, 128-byte swizzle: chunk index ^ (r & 7)
                const int chunk = (kh * 4 + j) ^ (r & 7);
                const int off = r * 128 + chunk * 16;
                *reinterpret_cast<uint4*>(stage + C::OFF_PLANES + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4*>(stage + C::OFF_PLANES + C::PLANE + off) =
                    make_uint4(pm[0], pm[1], pm[2], pm[3]);
                *reinterpret_cast<uint4*>(stage + C::OFF_PLANES + 2 * C::PLANE + off) =
                    make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_CONV + s));
        }
        if (ok) ok = __all_sync(kFull, mbar_wait(bar(B_ACC), 0, abort_flag, st, kSiteEpiAcc2Full));
        if (ok) {
            tc_fence_after();
            const int q = warp & 3;
            const int t = t0 + q * 32 + lane;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
            for (int c16 = 0; c16 < C::BN / 16; ++c16) {
                uint32_t v[16];
                tmem_ld16(taddr + c16 * 16, v);
                tmem_ld_wait();
                if (t < T) {
                    float4* dst = reinterpret_cast<float4*>(logits + static_cast<size_t>(t) * N + n0 + c16 * 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::BN);
    }
}

// The tensor-core router applies to bf16 tokens with H % 64 == 0, N % 64 == 0
// and 16-byte aligned logits.
static bool router_tc_ok(int x_dtype, int H, int N, const float* logits) {
    return x_dtype == MOE_DTYPE_BF16 && H % RtCfg::BK == 0 && N % RtCfg::BN == 0 &&
           (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
}

static cudaError_t launch_router_tc(const void* x, const float* w_router, int T, int H, int N, float* logits,
                                    moe_dev_status* st, cudaStream_t s) {
    using C = RtCfg;
    CUtensorMap tm_x, tm_w;
    if (!make_tmap(&tm_x, x, H, static_cast<uint64_t>(T), C::BK, C::BM) ||
        !make_tmap_f32(&tm_w, w_router, H, static_cast<uint64_t>(N), C::BK, C::BN))
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid((T + C::BM - 1) / C::BM, N / C::BN);
    return launch_pdl(router_tc_kernel, grid, dim3(C::THREADS), C::SMEM, s, tm_x, tm_w, T, H, N, logits, st);
}

cudaError_t launch_router(const void* x, int x_dtype, const float* w_router, int T, int H, int N, float* logits,
                          moe_dev_status* st, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (T > kRouterTcMinT && router_tc_ok(x_dtype, H, N, logits))
        return launch_router_tc(x, w_router, T, H, N, logits, st, s);
    if (T <= 256) {
        dim3 grid((N + 1) / 2, (T + 3) / 4);
        if (x_dtype == MOE_DTYPE_BF16)
            return launch_pdl(router_warp_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                              static_cast<const __nv_bfloat16*>(x), w_router, T, H, N, logits);
        return launch_pdl(router_warp_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(x), w_router, T,
                          H, N, logits);
    } else {
        dim3 grid((N + 63) / 64, (T + 63) / 64);
        if (x_dtype == MOE_DTYPE_BF16)
            return launch_pdl(router_tiled_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                              static_cast<const __nv_bfloat16*>(x), w_router, T, H, N, logits);
        return launch_pdl(router_tiled_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(x), w_router,
                          T, H, N, logits);
    }
    return cudaGetLastError();
}

constexpr int kSereStageN = 128;  // sim staged in shared memory up to N = 128 (64 KiB + N bytes)

template <int PL>
__global__ void __launch_bounds__(256) rank_kernel(const float* __restrict__ logits, int T, int N, int R, int k,
                                                   int renorm, int32_t* __restrict__ ids,
                                                   float* __restrict__ gates, moe_dev_status* st) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int id;
    float g;
    const bool ok = rank_token<PL>(logits + static_cast<size_t>(t) * N, N, R, k, renorm != 0, id, g);
    if (!ok && lane == 0) report(st, MOE_DEV_NONFINITE, t);
    if (lane < R) {
        ids[static_cast<size_t>(t) * R + lane] = id;
        gates[static_cast<size_t>(t) * R + lane] = g;
    }
}

template <int PL>
static cudaError_t rank_launch(const float* logits, int T, int N, int R, int k, bool renorm, int32_t* ids,
                               float* gates, moe_dev_status* st, cudaStream_t s) {
    return launch_pdl(rank_kernel<PL>, dim3((T + 7) / 8), dim3(256), 0, s, logits, T, N, R, k, renorm ? 1 : 0, ids,
                      gates, st);
}

cudaError_t launch_rank(const float* logits, int T, int N, int R, int k, bool renorm, int32_t* ids, float* gates,
                        moe_dev_status* st, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (N <= 32) return rank_launch<1>(logits, T, N, R, k, renorm, ids, gates, st, s);
    if (N <= 64) return rank_launch<2>(logits, T, N, R, k, renorm, ids, gates, st, s);
    if (N <= 128) return rank_launch<4>(logits, T, N, R, k, renorm, ids, gates, st, s);
    return rank_launch<8>(logits, T, N, R, k, renorm, ids, gates, st, s);
}

// ---------------------------------------------------------------------------
// The fused routing kernel: one thread-block cluster of CL CTAs (8 warps each)
// handles the whole batch.  Each CTA ranks its share of the tokens, the
// primary union P is OR-ed across the cluster through distributed shared
// memory, each CTA reroutes its own tokens against P, and CTA 0 gathers the
// after-union and the statistics.  Cluster barriers are hardware barriers; no
// host synchronisation and no sort.  Each CTA streams the similarity matrix
// into its shared memory with one bulk copy issued at the start, which lands
// while the tokens are being ranked.
// ---------------------------------------------------------------------------
namespace cg = cooperative_groups;
constexpr int kSereWarps = 8;

template <int PL>
__global__ void __launch_bounds__(256, 1) rank_sere_kernel(const float* __restrict__ logits, int do_rank, int T,
                                                           int N, int k, int renorm, int32_t* __restrict__ ids,
                                                           float* __restrict__ gates, int ld, int kp, float rho,
                                                           const float* __restrict__ sim,
                                                           const uint8_t* __restrict__ protect,
                                                           uint32_t* __restrict__ union_bitmap,
                                                           int32_t* __restrict__ stats, moe_dev_status* st,
                                                           int stage_sim) {
    __shared__ uint32_t Ploc[kMaxPerLane], Pall[kMaxPerLane], Ubefore[kMaxPerLane], Uafter[kMaxPerLane];
    __shared__ int sstats[8];
    __shared__ __align__(8) uint64_t sim_bar;
    __shared__ int abort_flag;
    extern __shared__ float4 s_sim4[];  // [N][N] fp32 similarity then [N] protect bytes, when staged
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(cluster.block_rank());
    const int csize = static_cast<int>(cluster.num_blocks());
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gwarp = crank * kSereWarps + warp, nwarps = csize * kSereWarps;
    const int n4 = (N * N) / 4;
    bool staged = stage_sim != 0;
    if (threadIdx.x < kMaxPerLane) {
        Ploc[threadIdx.x] = 0u;
        Ubefore[threadIdx.x] = 0u;
        Uafter[threadIdx.x] = 0u;
    }
    if (threadIdx.x < 8) sstats[threadIdx.x] = 0;
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (staged) {
            mbar_init(smem_u32(&sim_bar), 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(smem_u32(&sim_bar), static_cast<uint32_t>(n4) * 16u);
            bulk_copy_g2s(smem_u32(s_sim4), sim, static_cast<uint32_t>(n4) * 16u, smem_u32(&sim_bar));
        }
    }
    uint8_t* sprot = reinterpret_cast<uint8_t*>(s_sim4 + n4);
    if (staged && protect != nullptr)
        for (int i = threadIdx.x; i < N; i += blockDim.x) sprot[i] = protect[i];
    __syncthreads();
    // with at most one token per warp the routing stays in registers between the phases
    const bool in_regs = T <= nwarps;
    int id = -1;
    float g = 0.f;
    for (int t = gwarp; t < T; t += nwarps) {
        id = -1;
        g = 0.f;
        if (do_rank) {
            const bool ok = rank_token<PL>(logits + static_cast<size_t>(t) * N, N, k, k, renorm != 0, id, g);
            if (!ok && lane == 0) report(st, MOE_DEV_NONFINITE, t);
            if (!in_regs && lane < k) {
                ids[static_cast<size_t>(t) * ld + lane] = id;
                gates[static_cast<size_t>(t) * ld + lane] = g;
            }
        } else if (lane < k) {
            id = ids[static_cast<size_t>(t) * ld + lane];
            g = gates[static_cast<size_t>(t) * ld + lane];
        }
        if (lane < k && id >= N) {
            report(st, MOE_DEV_BAD_INDEX, id);
            id = -1;
        }
        if (lane < k && id >= 0) {
            atomicOr(&Ubefore[id >> 5], 1u << (id & 31));
            if (lane < kp) atomicOr(&Ploc[id >> 5], 1u << (id & 31));
        }
    }
    cluster.sync();  // every CTA's local primaries are in its shared memory
    if (threadIdx.x < kMaxPerLane) {
        uint32_t v = 0u;
        for (int r = 0; r < csize; ++r) v |= cluster.map_shared_rank(Ploc, r)[threadIdx.x];
        Pall[threadIdx.x] = v;
    }
    if (staged) {
        // every thread observes the copy's completion (bounded); on a time-out
        // the kernel records it and reads the similarity from global memory
        if (!mbar_wait(smem_u32(&sim_bar), 0, &abort_flag, st, kSiteDrain)) staged = false;
    }
    staged = __syncthreads_and(staged ? 1 : 0) != 0;
    const float* simp = staged ? reinterpret_cast<const float*>(s_sim4) : sim;
    const uint8_t* protp = (staged && protect != nullptr) ? sprot : protect;
    for (int t = gwarp; t < T; t += nwarps) {
        if (!in_regs) {
            id = -1;
            g = 0.f;
            if (lane < k) {
                id = ids[static_cast<size_t>(t) * ld + lane];
                g = gates[static_cast<size_t>(t) * ld + lane];
                if (id >= N) id = -1;
            }
        }
        sere_token<PL>(N, k, kp, rho, simp, protp, Pall, id, g, sstats);
        if (lane < k) {
            ids[static_cast<size_t>(t) * ld + lane] = id;
            gates[static_cast<size_t>(t) * ld + lane] = g;
            if (id >= 0) atomicOr(&Uafter[id >> 5], 1u << (id & 31));
        }
    }
    cluster.sync();  // every CTA's after-union and counters are final
    if (crank == 0) {
        if (threadIdx.x < kMaxPerLane) {
            uint32_t ub = 0u, ua = 0u;
            for (int r = 0; r < csize; ++r) {
                ub |= cluster.map_shared_rank(Ubefore, r)[threadIdx.x];
                ua |= cluster.map_shared_rank(Uafter, r)[threadIdx.x];
            }
            Ubefore[threadIdx.x] = ub;   // safe: the other CTAs read only Ploc from this CTA
            Uafter[threadIdx.x] = ua;
            if (union_bitmap != nullptr && threadIdx.x < (N + 31) / 32) union_bitmap[threadIdx.x] = Pall[threadIdx.x];
        } else if (threadIdx.x >= 32 && threadIdx.x < 40) {
            const int i = threadIdx.x - 32;
            int v = 0;
            for (int r = 0; r < csize; ++r) v += cluster.map_shared_rank(sstats, r)[i];
            sstats[i] = v;   // only CTA 0's own copy is rewritten, after every remote read of it
        }
    }
    if (stage_sim != 0 && !staged && threadIdx.x == 0) {
        // the copy did not complete in time: let it land before this CTA's shared memory is released
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(smem_u32(&sim_bar), 0) && global_ns() - t0 < kWaitLimitNs) {
        }
    }
    __syncthreads();
    if (crank == 0 && threadIdx.x == 0 && stats != nullptr) {
        int ub = 0, np = 0, ua = 0;
        for (int w = 0; w < kMaxPerLane; ++w) {
            ub += __popc(Ubefore[w]);
            np += __popc(Pall[w]);
            ua += __popc(Uafter[w]);
        }
        stats[0] = ub;
        stats[1] = np;
        stats[2] = ua;
        for (int i = 3; i < 7; ++i) stats[i] = sstats[i];
        stats[7] = 0;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

template <int PL>
static cudaError_t sere_launch_pl(const float* logits, int do_rank, int T, int N, int k, bool renorm, int32_t* ids,
                                  float* gates, int ld, const moe_sere_params& p, moe_dev_status* st, cudaStream_t s,
                                  bool stage, size_t smem, int csize) {
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(rank_sere_kernel<PL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSereStageN * kSereStageN * 4 + kSereStageN + 16));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize);
    cfg.blockDim = dim3(32 * kSereWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int renorm_i = renorm ? 1 : 0, stage_i = stage ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, rank_sere_kernel<PL>, logits, do_rank, T, N, k, renorm_i, ids, gates, ld,
                              p.k_primary, p.rho, p.sim, p.protect, p.union_bitmap, p.stats, st, stage_i);
}

// Stages sim in shared memory when it fits and can be copied with 16-byte
// transfers; the cluster has one CTA per 8 tokens, at most 8 CTAs.
static cudaError_t sere_launch(const float* logits, int do_rank, int T, int N, int k, bool renorm, int32_t* ids,
                               float* gates, int ld, const moe_sere_params& p, moe_dev_status* st, cudaStream_t s) {
    const bool stage = N <= kSereStageN && (N % 2) == 0 && (reinterpret_cast<uintptr_t>(p.sim) & 15u) == 0;
    const size_t smem = stage ? (static_cast<size_t>(N) * N * 4 + N + 15) / 16 * 16 : 0;
    int csize = (T + kSereWarps - 1) / kSereWarps;
    csize = csize < 1 ? 1 : (csize > 8 ? 8 : csize);
    if (N <= 32) return sere_launch_pl<1>(logits, do_rank, T, N, k, renorm, ids, gates, ld, p, st, s, stage, smem, csize);
    if (N <= 64) return sere_launch_pl<2>(logits, do_rank, T, N, k, renorm, ids, gates, ld, p, st, s, stage, smem, csize);
    if (N <= 128) return sere_launch_pl<4>(logits, do_rank, T, N, k, renorm, ids, gates, ld, p, st, s, stage, smem, csize);
    return sere_launch_pl<8>(logits, do_rank, T, N, k, renorm, ids, gates, ld, p, st, s, stage, smem, csize);
}

cudaError_t launch_rank_sere(const float* logits, int T, int N, int k, bool renorm, int32_t* ids, float* gates,
                             const moe_sere_params& p, moe_dev_status* st, cudaStream_t s) {
    return sere_launch(logits, 1, T, N, k, renorm, ids, gates, k, p, st, s);
}

cudaError_t launch_sere(int32_t* ids, float* gates, int ld, int T, int N, int k, const moe_sere_params& p,
                        moe_dev_status* st, cudaStream_t s) {
    return sere_launch(nullptr, 0, T, N, k, false, ids, gates, ld, p, st, s);
}

}  // namespace moe
