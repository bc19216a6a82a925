// One-shot all-reduce, emulated on one device in a single cooperative launch.
//
// memra-engine 0.128.0 tests/tp_ar_gpu.rs (`one_shot_all_reduce_matches_the_
// host_sum_bitwise`) describes the shape: one kernel per rank and no events,
// a device barrier on entry and on exit whose expiry returns with x untouched
// and sets a refusal word (40043 entry, 40044 exit), and repeat calls that
// must keep working. Here the W ranks are W groups of CTAs of one launch, so
// they are co-resident by construction (cooperative launch), and every rank
// group reads all W arenas directly:
//
//   1. entry barrier: every CTA publishes the call's epoch in its own flag
//      (release) and waits, bounded, until every CTA's flag has it (acquire);
//   2. rank r folds all arenas in ascending rank order (mamba-rs 0.6.2
//      src/dist/reducer.rs, `reduce_sum_reference`) into its stage row, times
//      the mean scale;
//   3. exit barrier, the same on the exit flags: nobody is still reading x;
//   4. rank r copies its stage row into its arena.
//
// Waits are bounded by %globaltimer (wait_ns) and by an iteration cap; an
// expired wait writes the rank's refusal word and returns before step 4, so
// the arena keeps its old contents. Epoch flags only grow, so a call that
// refused leaves nothing to reset: the next call's larger epoch starts clean.
//
// The epoch comes from the host (>= 1) or, when the host passes 0, from a
// counter in the link: every CTA reads it before publishing anything and uses
// counter + 1. Every CTA that ran raises the counter to its epoch (atomicMax)
// on each way out, so the next call starts above every flag ever published,
// also after refused calls. In a call that completes, all CTAs read the
// counter before any of them passes the exit barrier and raises it, so they
// agree on the epoch. A captured graph therefore replays correctly: each
// replay takes the next epoch from device memory.
// For failure-detection tests the host may drop one rank at the entry or the
// exit barrier (it never publishes there), which makes the others' waits run
// out by design.
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold.h"
#include "detfold_launch.cuh"

namespace detfold {

namespace {

constexpr int kOneShotThreads = 256;
constexpr unsigned kMaxPolls = 1u << 26;  // hard cap on polls of one wait
constexpr int kU = 4;                     // elements per thread per group
constexpr int kFastW = 8;                 // worlds up to this size load a group ahead

struct OneShotParams {
    float *arena[DETFOLD_ONESHOT_MAX_W];
    float *stage;                      // W rows of len floats
    unsigned long long *entry_flags;   // DETFOLD_ONESHOT_MAX_CTAS each
    unsigned long long *exit_flags;
    unsigned long long *counter;       // the link's epoch counter
    int *words;                        // W refusal words
    unsigned long long epoch;          // 0: counter + 1
    int64_t len;
    long long wait_ns;
    float scale;
    int do_scale;
    int W;
    int ctas_per_rank;
    int drop_rank;                     // -1: nobody dropped
    int drop_at_exit;                  // 0: the dropped rank skips the entry barrier
};

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ long long global_ns()
{
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Publish this CTA's arrival and wait (bounded) for every CTA's. Returns
// false if the wait ran out. All threads of the CTA call it.
__device__ bool cta_barrier(unsigned long long *flags, int nctas, unsigned long long epoch,
                            long long wait_ns, bool publish)
{
    __shared__ int s_ok;
    __syncthreads();  // this CTA's earlier writes are done
    if (threadIdx.x == 0) {
        __threadfence();
        if (publish) st_release(flags + blockIdx.x, epoch);
    }
    if (threadIdx.x < 32) {
        const long long t0 = global_ns();
        bool ok = false;
        for (unsigned poll = 0; poll < kMaxPolls; ++poll) {
            bool mine = true;
            for (int b = threadIdx.x; b < nctas; b += 32) mine = mine && ld_acquire(flags + b) >= epoch;
            if (__all_sync(0xffffffffu, mine)) {
                ok = true;
                break;
            }
            // the expiry decision must be the same in every lane of the warp
            if (__any_sync(0xffffffffu, global_ns() - t0 > wait_ns)) break;
            __nanosleep(32);
        }
        if (threadIdx.x == 0) s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ void raise_counter(const OneShotParams &p, unsigned long long epoch)
{
    if (threadIdx.x == 0) atomicMax(p.counter, epoch);
}

__global__ void __launch_bounds__(kOneShotThreads) one_shot_kernel(const __grid_constant__ OneShotParams p)
{
    const int r = blockIdx.x / p.ctas_per_rank;
    const int g = blockIdx.x % p.ctas_per_rank;
    const int nctas = gridDim.x;
    const bool dropped = (r == p.drop_rank);
    __shared__ unsigned long long s_epoch;
    if (threadIdx.x == 0) s_epoch = p.epoch ? p.epoch : ld_acquire(p.counter) + 1;
    __syncthreads();
    const unsigned long long epoch = s_epoch;
    if (g == 0 && threadIdx.x == 0) p.words[r] = DETFOLD_OK;  // a dropped rank refuses nothing

    // 1. entry barrier
    if (dropped && !p.drop_at_exit) {  // this rank never joins
        raise_counter(p, epoch);
        return;
    }
    if (!cta_barrier(p.entry_flags, nctas, epoch, p.wait_ns, true)) {
        if (g == 0 && threadIdx.x == 0) p.words[r] = DETFOLD_ONESHOT_REFUSE_ENTRY;
        raise_counter(p, epoch);
        return;  // x untouched
    }

    // 2. rank r folds every arena into its stage row (its CTAs split the
    // row). A thread's elements i, i + stride, ... go kU at a time; up to
    // kFastW ranks, every load of the group is issued before the first add
    // (one memory round trip per group, not one per element). The chain of
    // each element stays in ascending rank order.
    float *stage = p.stage + (int64_t)r * p.len;
    const int64_t stride = (int64_t)p.ctas_per_rank * blockDim.x;
    for (int64_t i0 = (int64_t)g * blockDim.x + threadIdx.x; i0 < p.len; i0 += kU * stride) {
        if (p.W <= kFastW) {
            float x[kU][kFastW];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = i0 + u * stride;
#pragma unroll
                for (int q = 0; q < kFastW; ++q)
                    if (q < p.W && i < p.len) x[u][q] = ld1<false>(p.arena[q] + i);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = i0 + u * stride;
                if (i < p.len) {
                    float acc = x[u][0];
#pragma unroll
                    for (int q = 1; q < kFastW; ++q)
                        if (q < p.W) acc = __fadd_rn(acc, x[u][q]);
                    if (p.do_scale) acc = __fmul_rn(acc, p.scale);
                    st1(stage + i, acc);
                }
            }
        } else {
            for (int u = 0; u < kU; ++u) {
                const int64_t i = i0 + u * stride;
                if (i < p.len) {
                    float acc = ld1<false>(p.arena[0] + i);
                    for (int q = 1; q < p.W; ++q) acc = __fadd_rn(acc, ld1<false>(p.arena[q] + i));
                    if (p.do_scale) acc = __fmul_rn(acc, p.scale);
                    st1(stage + i, acc);
                }
            }
        }
    }

    // 3. exit barrier: every rank has finished reading the arenas
    if (dropped) {  // dropped at the exit barrier: never publishes there
        raise_counter(p, epoch);
        return;
    }
    if (!cta_barrier(p.exit_flags, nctas, epoch, p.wait_ns, true)) {
        if (g == 0 && threadIdx.x == 0) p.words[r] = DETFOLD_ONESHOT_REFUSE_EXIT;
        raise_counter(p, epoch);
        return;  // x untouched
    }

    // 4. the stage row becomes the arena (the elements this thread staged,
    // kU loads ahead of their stores)
    for (int64_t i0 = (int64_t)g * blockDim.x + threadIdx.x; i0 < p.len; i0 += kU * stride) {
        float y[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (i0 + u * stride < p.len) y[u] = ld1<false>(stage + i0 + u * stride);
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (i0 + u * stride < p.len) st1(p.arena[r] + i0 + u * stride, y[u]);
    }
    raise_counter(p, epoch);
}

}  // namespace

cudaError_t launch_one_shot(float *const *arenas, int W, int64_t len, float scale, int do_scale,
                            void *link, unsigned long long epoch, float *stage, int *words,
                            long long wait_ns, int drop_rank, int drop_at_exit,
                            cudaStream_t stream);

cudaError_t launch_one_shot(float *const *arenas, int W, int64_t len, float scale, int do_scale,
                            void *link, unsigned long long epoch, float *stage, int *words,
                            long long wait_ns, int drop_rank, int drop_at_exit,
                            cudaStream_t stream)
{
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, one_shot_kernel, kOneShotThreads, 0);
    if (e != cudaSuccess) return e;
    // every CTA must be resident at once: the cooperative launch refuses otherwise
    const int64_t resident = (int64_t)sms * per_sm;
    int64_t per_rank = (len + 4 * kOneShotThreads - 1) / (4 * kOneShotThreads);
    if (per_rank > 8) per_rank = 8;
    if (per_rank < 1) per_rank = 1;
    while (per_rank > 1 && per_rank * W > resident) --per_rank;
    if (per_rank * W > resident || per_rank * W > DETFOLD_ONESHOT_MAX_CTAS) return cudaErrorCooperativeLaunchTooLarge;

    OneShotParams p = {};
    for (int r = 0; r < W; ++r) p.arena[r] = arenas[r];
    p.stage = stage;
    p.entry_flags = (unsigned long long *)link;
    p.exit_flags = (unsigned long long *)link + DETFOLD_ONESHOT_MAX_CTAS;
    p.counter = (unsigned long long *)link + 2 * DETFOLD_ONESHOT_MAX_CTAS;
    p.words = words;
    p.epoch = epoch;
    p.len = len;
    p.wait_ns = wait_ns;
    p.scale = scale;
    p.do_scale = do_scale;
    p.W = W;
    p.ctas_per_rank = (int)per_rank;
    p.drop_rank = drop_rank;
    p.drop_at_exit = drop_at_exit;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(per_rank * W), 1, 1);
    cfg.blockDim = dim3(kOneShotThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, one_shot_kernel, p);
}

}  // namespace detfold
