// cast.cu -- the residual stream's fp32 -> bf16 rounding between stacked MoE
// layers.  A layer adds sum_j G_j E_j(x) into the fp32 residual (the FFN's
// accumulate mode); the next layer routes and gathers bf16 rows, so the
// residual is rounded (to nearest, ties to even) once per layer.  The
// launch uses programmatic dependent launch like every kernel of the
// library, so it overlaps the FFN's tail and the next routing launch
// overlaps it.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"   // sm_count

namespace moe {

// Eight elements per thread: two 16-byte loads, one 16-byte store.
__global__ void __launch_bounds__(256) residual_to_bf16_kernel(const float4* __restrict__ x,
                                                               uint4* __restrict__ y, long long n8) {
    pdl_wait();
    pdl_trigger();
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = x[2 * i], b = x[2 * i + 1];
        const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
        y[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                          *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
    }
}

cudaError_t launch_residual_to_bf16(const float* x, void* y, long long n, cudaStream_t s) {
    const long long n8 = n / 8;
    long long grid = (n8 + 255) / 256;
    const long long cap = 4ll * sm_count();
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_pdl(residual_to_bf16_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                      reinterpret_cast<const float4*>(x), static_cast<uint4*>(y), n8);
}

}  // namespace moe
