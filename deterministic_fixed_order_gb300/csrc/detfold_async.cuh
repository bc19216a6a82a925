// Bulk-async (TMA) building blocks for the staged pipelines: mbarrier
// set-up, arrival and bounded waits, cp.async.bulk loads (global -> shared,
// completion by byte count on an mbarrier) and stores (shared -> global, in
// bulk groups), and the proxy fence between generic shared-memory writes and
// a bulk store. Every wait is bounded; an expiry is counted in
// g_pipeline_timeouts. Each translation unit that includes this header has
// its own counter (internal linkage: device code is compiled per unit) and
// exports a reader; detfold_pipeline_timeouts sums them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace detfold {

static __device__ unsigned long long g_pipeline_timeouts;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ long long now_ns()
{
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.
static __device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity)
{
    const long long t0 = now_ns();
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try(b, parity)) return true;
        if (now_ns() - t0 > 1000000000LL) break;
    }
    atomicAdd(&g_pipeline_timeouts, 1ull);
    return false;
}

#ifndef DETFOLD_BULK_L2_HINT
#define DETFOLD_BULK_L2_HINT 0  // 1: loads evict-first in L2, 2: stores, 3: both
#endif

// An L2 cache policy that marks lines for early eviction (streamed once).
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
#if DETFOLD_BULK_L2_HINT & 1
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(evict_first_policy())
        : "memory");
    return;
#endif
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
#if DETFOLD_BULK_L2_HINT & 2
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes), "l"(evict_first_policy())
                 : "memory");
    return;
#endif
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier of n threads that also ORs one predicate over them: every
// participant gets the same answer. A group whose members each ran their own
// bounded wait meets here and takes one verdict, so no member can leave
// while another still waits at a later barrier for it. Same memory ordering
// as bar.sync.
__device__ __forceinline__ bool named_sync_any(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
        " selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

#ifndef DETFOLD_BULK_EXCLUSIVE
#define DETFOLD_BULK_EXCLUSIVE 1  // 1: bulk CTAs reserve shared memory so no SM holds more than planned
#endif

// Host side. Dynamic shared memory to request per CTA of a grid planned for
// `per_sm` CTAs on every SM: the kernel's own need, raised (when
// DETFOLD_BULK_EXCLUSIVE) until a (per_sm + 1)-th CTA no longer fits on an
// SM. The bulk kernels give every CTA a fixed share of the tiles, so an SM
// holding an extra CTA would finish last. That happens when programmatic
// dependent launch places CTAs while the previous kernel still occupies the
// SMs: measured on GB300, a W=4 all-reduce planned for 2 CTAs per SM in
// 41 KB each (5 fit) cost a back-to-back step 0.25 ms more than the same
// kernel run alone.
static inline cudaError_t exclusive_smem(int dev, size_t need, int per_sm, size_t *out)
{
    *out = need;
    if (!DETFOLD_BULK_EXCLUSIVE || per_sm <= 0) return cudaSuccess;
    int per_sm_bytes = 0, reserved = 0, optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&per_sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    // (per_sm + 1) * (x + reserved) > per_sm_bytes, rounded up to 128 bytes
    size_t x = (size_t)(per_sm_bytes / (per_sm + 1) - reserved + 1);
    x = (x + 127) / 128 * 128;
    if (x > need && x <= (size_t)optin && (size_t)per_sm * (x + reserved) <= (size_t)per_sm_bytes) *out = x;
    return cudaSuccess;
}

// Host side: this translation unit's counter.
static inline cudaError_t read_unit_timeouts(unsigned long long *count)
{
    return cudaMemcpyFromSymbol(count, g_pipeline_timeouts, sizeof(*count));
}

}  // namespace detfold
