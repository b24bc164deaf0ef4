// common.cuh -- shared device helpers of the GB300 MoE library: status
// reporting, deterministic fp32 arithmetic for the gate, bounded waits and
// the sm_103a inline-PTX wrappers (mbarrier, TMA, tcgen05).
#pragma once

#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// Wait sites reported in moe_dev_status.detail on MOE_DEV_TIMEOUT.
enum WaitSite : int {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaTmemFree = 3,
    kSiteMmaActReady = 4,
    kSiteMmaAcc2Empty = 5,
    kSiteEpiG1Done = 6,
    kSiteEpiActFree = 7,
    kSiteEpiAcc2Full = 8,
    kSiteDrain = 9,
    kSiteDependency = 10,
};

// Longest time a single on-chip wait may take before the kernel gives up
// (ns).  Legitimate waits in these kernels last microseconds.
constexpr unsigned long long kWaitLimitNs = 1500000000ull;

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible (a no-op without a
// programmatic dependency), and allow the next kernel to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void report(moe_dev_status* st, int code, int detail) {
    if (st == nullptr) return;
    if (atomicCAS(&st->code, 0, code) == 0) atomicExch(&st->detail, detail);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Deterministic fp32 exponential for d <= 0, used for the softmax gate.
// Cody & Waite reduction d = n ln2 + r with a 15-bit head of ln2 (n*ln2_hi is
// exact for |n| < 512), the degree-7 Taylor polynomial of e^r evaluated with
// fused multiply-adds, and an exact scaling by 2^n; results that would be
// below 2^-125 flush to zero.  Every operation is an explicitly rounded
// intrinsic, so the compiler cannot contract or reorder it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_gate(float d) {
    const float log2e = 0x1.715476p+0f;     // log2(e), nearest fp32
    const float ln2_hi = 0x1.62e4p-1f;      // 22713 / 2^15
    const float ln2_lo = 0x1.7f7d1cp-20f;   // ln2 - ln2_hi, nearest fp32
    float n = rintf(__fmul_rn(d, log2e));
    if (n < -125.0f) return 0.0f;
    float r = __fmaf_rn(-n, ln2_hi, d);
    r = __fmaf_rn(-n, ln2_lo, r);
    // 1/i! for i = 7 .. 0, nearest fp32
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1p-1f);
    p = __fmaf_rn(p, r, 0x1p+0f);
    p = __fmaf_rn(p, r, 0x1p+0f);
    const int ni = static_cast<int>(n);
    return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// Orders (value, id) pairs: larger value first, then lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Warp-wide best (value, id) under ranks_before.  Ids < 0 mean "none".
__device__ __forceinline__ void warp_best(float& v, int& id) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        float ov = __shfl_xor_sync(kFull, v, off);
        int oi = __shfl_xor_sync(kFull, id, off);
        bool take = (oi >= 0) && (id < 0 || ranks_before(ov, oi, v, id));
        if (take) { v = ov; id = oi; }
    }
}

// ---------------------------------------------------------------------------
// Shared-memory address helpers and mbarrier wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// when `abort_flag` becomes nonzero or after kWaitLimitNs; on time-out it sets
// the abort flag and reports the wait site.  Returns true on success.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          moe_dev_status* st, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            report(st, MOE_DEV_TIMEOUT, site);
            return false;
        }
    }
}

// Waits (bounded, ignoring the abort flag) for a phase that must complete
// before shared memory or TMEM is released, e.g. copies still in flight.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  x = innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk (non-tensor) copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completion signalled on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Prefetch one 2-D box of a tensor into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy accesses to global memory with its
// later (or earlier) async-proxy ones, e.g. TMA loads of data that another
// CTA stored with plain st.global.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Ticket: fetch-and-add with acquire-release semantics at GPU scope.  Taken
// by one thread after a CTA barrier, it publishes the CTA's earlier writes
// and, for the CTA that draws the last ticket, makes every other CTA's
// published writes visible to the reads after its next barrier.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Named barrier 1 over `nthreads` threads (whole warps) that returns the AND
// of every participant's `v`.  Callers pass it the same number of times in
// every participating warp, so that a failed wait in one warp cannot strand
// the others at a barrier: they all learn of it here and leave together.
__device__ __forceinline__ bool named_sync_and(int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------
// tcgen05 wrappers (5th-generation tensor cores, accumulators in TMEM).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp gets lane
// (quadrant base + i), columns [col, col+16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}

// TMA gather of four rows (tensor map box: 64 columns x 1 row) into four
// consecutive 128-byte rows of shared memory.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int x, int r0, int r1, int r2, int r3,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle (rows of 64 bf16 = 128 B, 8-row atoms of 1024 B).
// Fields: start address >> 4 [0,14); leading byte offset >> 4 [16,30)
// (unused for swizzled K-major, set to 1); stride byte offset >> 4 [32,46)
// = 1024 B between 8-row groups; descriptor version 1 [46,48); base offset 0
// (tiles are 1024-byte aligned); layout type 2 = SWIZZLE_128B [61,64).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both K-major.
// Fields: D format [4,6) = 1 (f32); A format [7,10) = 1 (bf16); B format
// [10,13) = 1 (bf16); transpose bits 15/16 = 0 (K-major); N >> 3 at [17,23);
// M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace moe
