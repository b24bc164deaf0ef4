// calib.cu -- expert similarity from calibration tokens.
//
// Xiaohongshu multi-image QA inference article, sec. 4.2: the SERE
// similarity matrix is computed offline as the Frobenius similarity of the
// experts' outputs on calibration data,
//   sim[i][j] = <E_i(X), E_j(X)>_F / (||E_i(X)||_F ||E_j(X)||_F),
// E_e(X) the [n][H] outputs of expert e ("MACS" Eq. (1)'s E_j) on the n
// calibration tokens.
//
// 1. Every token goes to every expert: the permutation is built directly
//    (row e*n + t = token t at expert e) and the grouped tcgen05 FFN writes
//    E_e(x_t) for all n*N rows (rows_out mode, fp32).
// 2. The rows are rounded to bf16; viewed as an [N][n*H] matrix (rows are
//    expert-major) they give G = E E^T on the tensor cores: each CTA takes a
//    K range, TMA brings 128 x 64 tiles, one tcgen05 MMA per 16 columns uses
//    the same tile as both operands (D[128 x 128] in TMEM), and the CTA
//    stores its partial G.
// 3. The partials are summed in a fixed order and normalised in double.
// The rounding to bf16 perturbs each product by at most 2^-8 relative; over
// the n*H products of a similarity those errors average out to about 1e-5.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace moe {

constexpr int kCalibMaxN = 128;

struct CalibLayout {
    size_t offsets, active, row_token, row_gate, ffn, rows, ebf, partials, gram, total;
    int grid;
};

static size_t al256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

static CalibLayout calib_layout(int n, int H, int I, int N) {
    CalibLayout L;
    const size_t M = static_cast<size_t>(n) * N;
    L.grid = sm_count();
    size_t o = 0;
    L.offsets = o; o += al256((N + 1) * 4);
    L.active = o; o += al256((N + 1) * 4);
    L.row_token = o; o += al256(M * 4);
    L.row_gate = o; o += al256(M * 4);
    L.ffn = o; o += al256(ffn_workspace(n, H, I, N, N, MOE_DTYPE_BF16));
    L.rows = o; o += al256(M * H * 4);
    L.ebf = o; o += al256(M * H * 2);
    L.partials = o; o += al256(static_cast<size_t>(L.grid) * 128 * 128 * 4);
    L.gram = o; o += al256(static_cast<size_t>(N) * N * 8);
    L.total = o;
    return L;
}

size_t calib_workspace(int n, int H, int I, int N) {
    if (n < 1 || N > kCalibMaxN) return 0;
    return calib_layout(n, H, I, N).total;
}

// Every token to every expert; clears the fp32 row outputs (accumulated into).
__global__ void calib_perm_kernel(int n, int N, int H, int32_t* offsets, int32_t* active, int32_t* row_token,
                                  float* row_gate, float4* rows4) {
    pdl_wait();
    pdl_trigger();
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long M = static_cast<long long>(n) * N;
    for (long long r = tid; r < M; r += nthr) {
        row_token[r] = static_cast<int32_t>(r % n);
        row_gate[r] = 1.0f;
    }
    for (long long e = tid; e <= N; e += nthr) {
        offsets[e] = static_cast<int32_t>(e * n);
        active[e] = (e == 0) ? N : static_cast<int32_t>(e - 1);
    }
    const long long n4 = M * H / 4;
    for (long long i = tid; i < n4; i += nthr) rows4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void calib_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, long long n4) {
    pdl_wait();
    pdl_trigger();
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 v = in[i];
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
}

// Gram partials: CTA c accumulates D = A A^T over K chunks [c0, c1) of 64
// columns (A = the 128-row tile of E; rows >= N read as zero).
struct GramCfg {
    static constexpr int TILE = 128 * 64 * 2;   // 16 KiB
    static constexpr int NSTAGE = 4;
    static constexpr int THREADS = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
    static constexpr int SMEM = 1024 + NSTAGE * TILE + (2 * NSTAGE + 2) * 8 + 16;
};

__global__ void __launch_bounds__(GramCfg::THREADS, 1)
    calib_gram_kernel(const __grid_constant__ CUtensorMap tm_e, long long kchunks, float* __restrict__ partials,
                      moe_dev_status* st) {
    using C = GramCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::NSTAGE * C::TILE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::NSTAGE + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t ring_a = smem_u32(smem);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_FULL = 0, B_EMPTY = C::NSTAGE, B_ACC = 2 * C::NSTAGE, B_DRAIN = B_ACC + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long c0 = kchunks * blockIdx.x / gridDim.x, c1 = kchunks * (blockIdx.x + 1) / gridDim.x;
    const int nk = static_cast<int>(c1 - c0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_ACC), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_e);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 128);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            uint32_t pend = 0, pend_par = 0;
            bool ok = true;
            for (int c = 0; c < nk; ++c) {
                const int s = c % C::NSTAGE;
                const uint32_t ph = (c / C::NSTAGE) & 1;
                if (!mbar_wait(bar(B_EMPTY + s), ph ^ 1u, abort_flag, st, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(B_FULL + s), C::TILE);
                tma_load_2d(ring_a + s * C::TILE, &tm_e, static_cast<int>((c0 + c) * 64), 0, bar(B_FULL + s), pol);
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
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            bool ok = true;
            for (int c = 0; c < nk; ++c) {
                const int s = c % C::NSTAGE;
                if (!mbar_wait(bar(B_FULL + s), (c / C::NSTAGE) & 1, abort_flag, st, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = ring_a + s * C::TILE;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16(tmem, sw128_desc(a + kk * 32), sw128_desc(a + kk * 32), idesc, (c | kk) != 0);
                tc_commit(bar(B_EMPTY + s));
            }
            if (ok) tc_commit(bar(B_ACC));
            tc_commit(bar(B_DRAIN));
            mbar_drain(bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        float* dst = partials + (static_cast<size_t>(blockIdx.x) * 128 + row) * 128;
        if (nk == 0) {
            for (int j = 0; j < 128; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (__all_sync(kFull, mbar_wait(bar(B_ACC), 0, abort_flag, st, kSiteEpiAcc2Full))) {
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c16 = 0; c16 < 8; ++c16) {
                uint32_t v[16];
                tmem_ld16(taddr + c16 * 16, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<float4*>(dst + c16 * 16 + 4 * i) =
                        make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// G[i][j] = sum over CTAs (in order) of the partials, in double.
__global__ void calib_reduce_kernel(const float* __restrict__ partials, int nparts, int N, double* __restrict__ G) {
    pdl_wait();
    pdl_trigger();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * N) return;
    const int i = idx / N, j = idx % N;
    double s = 0.0;
    for (int p = 0; p < nparts; ++p) s += static_cast<double>(partials[(static_cast<size_t>(p) * 128 + i) * 128 + j]);
    G[idx] = s;
}

// sim[i][j] = G_ij / sqrt(G_ii G_jj) from the upper triangle (so sim is exactly
// symmetric); diagonal 1; 0 when either expert's output is all zero.
__global__ void calib_normalize_kernel(const double* __restrict__ G, int N, float* __restrict__ sim) {
    pdl_wait();
    pdl_trigger();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * N) return;
    const int i = idx / N, j = idx % N;
    const int a = min(i, j), b = max(i, j);
    float v = 1.0f;
    if (i != j) {
        const double gaa = G[static_cast<size_t>(a) * N + a], gbb = G[static_cast<size_t>(b) * N + b];
        v = (gaa > 0.0 && gbb > 0.0) ? static_cast<float>(G[static_cast<size_t>(a) * N + b] / sqrt(gaa * gbb))
                                     : 0.0f;
    }
    sim[idx] = v;
}

cudaError_t launch_similarity(const void* x, int n, const void* wg, const void* wu, const void* wd, int H, int I,
                              int N, float* sim, void* ws, moe_dev_status* st, cudaStream_t s) {
    const CalibLayout L = calib_layout(n, H, I, N);
    uint8_t* b = static_cast<uint8_t*>(ws);
    int32_t* offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    int32_t* active = reinterpret_cast<int32_t*>(b + L.active);
    int32_t* row_token = reinterpret_cast<int32_t*>(b + L.row_token);
    float* row_gate = reinterpret_cast<float*>(b + L.row_gate);
    float* rows = reinterpret_cast<float*>(b + L.rows);
    __nv_bfloat16* ebf = reinterpret_cast<__nv_bfloat16*>(b + L.ebf);
    float* partials = reinterpret_cast<float*>(b + L.partials);
    double* gram = reinterpret_cast<double*>(b + L.gram);
    const int sms = L.grid;
    const long long M = static_cast<long long>(n) * N;
    cudaError_t e = launch_pdl(calib_perm_kernel, dim3(4 * sms), dim3(256), 0, s, n, N, H, offsets, active, row_token,
                               row_gate, reinterpret_cast<float4*>(rows));
    if (e != cudaSuccess) return e;
    // E_e(x_t) for every expert and token: the grouped FFN with k = N, rows_out mode
    // (its counters start from zero; this workspace has no initial contents)
    e = cudaMemsetAsync(b + L.ffn, 0, ffn_workspace_zero_bytes(n, H, N, N, MOE_DTYPE_BF16), s);
    if (e != cudaSuccess) return e;
    e = launch_ffn_bf16(x, wg, wu, wd, n, H, I, N, N, offsets, row_token, row_gate, active, 0u, rows, b + L.ffn, st,
                        s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(calib_to_bf16_kernel, dim3(4 * sms), dim3(256), 0, s, reinterpret_cast<const float4*>(rows),
                   reinterpret_cast<uint2*>(ebf), M * H / 4);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_e;
    const long long K = static_cast<long long>(n) * H;
    if (!make_tmap(&tm_e, ebf, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 64, 128))
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[64] = {};   // per device; idempotent, race-free
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(calib_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GramCfg::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    e = launch_pdl(calib_gram_kernel, dim3(sms), dim3(GramCfg::THREADS), GramCfg::SMEM, s, tm_e, K / 64, partials,
                   st);
    if (e != cudaSuccess) return e;
    const int nn = N * N;
    e = launch_pdl(calib_reduce_kernel, dim3((nn + 255) / 256), dim3(256), 0, s, static_cast<const float*>(partials),
                   sms, N, gram);
    if (e != cudaSuccess) return e;
    return launch_pdl(calib_normalize_kernel, dim3((nn + 255) / 256), dim3(256), 0, s, static_cast<const double*>(gram),
                      N, sim);
}

}  // namespace moe
