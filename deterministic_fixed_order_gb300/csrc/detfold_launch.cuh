// Host-side launch plumbing shared by the mode translation units: phase
// planning (vector width, head, body, tail), grid sizing, the typed launch
// of one kernel instantiation, and the dispatch order of a fold call:
// bulk-async path (large, one 16-byte phase, W <= 8) -> small-payload kernel
// (small, common phase) -> vector kernel (common phase) -> the bulk-async
// all-reduce with per-arena offsets (large, mixed 16-byte phases) ->
// realigned vectors (mismatched phases).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold_kernels.cuh"

namespace detfold {

// One fold launch as the API layer describes it.
struct LaunchSpec {
    int W;
    int mode;                // Mode
    const float *const *src; // host array of W device pointers
    float *out;              // sum modes only
    int64_t len;
    float scale;
    int do_scale;
};

// How the elements are split: `vec` = 8, 4, or 0 for the scalar kernel.
struct Plan {
    int vec;
    int64_t head, nvec;
};

inline int elem_phase(const void *p, int vec)
{
    return (int)(((uintptr_t)p % (uintptr_t)(vec * 4)) / 4);
}

// The widest vector, at most `prefer` floats, whose phase every operand
// shares (the output as well).
inline Plan make_plan(const LaunchSpec &s, int prefer)
{
    const int prefs[2] = {prefer, 4};
    for (int k = 0; k < 2; ++k) {
        const int vec = prefs[k];
        const int ph = elem_phase(s.src[0], vec);
        bool same = (s.mode == kAllReduce) || elem_phase(s.out, vec) == ph;
        for (int r = 1; same && r < s.W; ++r) same = elem_phase(s.src[r], vec) == ph;
        if (same) {
            int64_t head = (vec - ph) % vec;
            if (head > s.len) head = s.len;
            return Plan{vec, head, (s.len - head) / vec};
        }
    }
    return Plan{0, 0, 0};
}

// Vectors (or scalars, vec == 0) per thread per unrolled group.
template <int MODE>
inline constexpr int u_for(int W, int vec)
{
    if (vec == 0) {
        const int u = DETFOLD_SCALAR_INFLIGHT / (4 * W);
        return u < 1 ? 1 : (u > DETFOLD_SCALAR_MAX_U ? DETFOLD_SCALAR_MAX_U : u);
    }
    // the W=1 scale pass goes deeper: at the C5 length (2^20 + 7) 512 bytes
    // per thread measured 2.07-2.13 us against 2.33-2.48 at 256
    const int bytes = MODE == kAllReduce ? (W == 1 ? DETFOLD_SCALE_INFLIGHT : DETFOLD_AR_INFLIGHT)
                                         : DETFOLD_SUM_INFLIGHT;
    int u = bytes / (vec * 4 * W);
    if (MODE != kAllReduce && u * W * vec > DETFOLD_SUM_MAX_FLOATS) u = DETFOLD_SUM_MAX_FLOATS / (W * vec);
    return u < 1 ? 1 : u;
}

// Resident CTAs the whole GPU holds for `Kernel` at `threads` per CTA (at
// most cap_per_sm per SM when cap_per_sm > 0). Computed once per kernel and
// device: the cache lives in this function's instantiation for that kernel.
template <auto Kernel>
inline cudaError_t resident_ctas(int threads, int cap_per_sm, int *out)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, Kernel, threads, 0);
        if (e != cudaSuccess) return e;
        if (cap_per_sm > 0 && per_sm > cap_per_sm) per_sm = cap_per_sm;
        v = sms * (per_sm > 0 ? per_sm : 1);
        cache[dev].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return cudaSuccess;
}

// Streaming multiprocessors of the current device, looked up once per device.
inline cudaError_t sm_count(int *out)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return cudaSuccess;
}

// One launch: the small path covers the work exactly with small CTAs; the
// bandwidth path runs a grid of at most the resident CTAs, each thread
// striding over U-vector groups. When the work would give fewer than
// DETFOLD_FILL_SMS CTAs per SM, the CTA size halves (down to 64 threads), so
// a medium-sized call spreads over every SM instead of a few large CTAs on
// some of them. Programmatic dependent launch is used exactly when the
// parameter block's pdl flag is set.
template <auto Kernel, typename Params>
inline cudaError_t launch_kernel(const Params &p, int64_t work, int u, bool small, int bw_threads,
                                 int cap_per_sm, cudaStream_t stream, bool fill = true,
                                 int extra_blocks = 0)
{
    int threads = small ? DETFOLD_SMALL_THREADS : bw_threads;
    int64_t blocks = (work + threads - 1) / threads;
    if (!small) {
        int64_t per_iter = (int64_t)threads * u;
        blocks = (work + per_iter - 1) / per_iter;
        int cap = 0;
        cudaError_t e = resident_ctas<Kernel>(threads, cap_per_sm, &cap);
        if (e != cudaSuccess) return e;
        if (DETFOLD_FILL_SMS > 0 && fill && blocks < cap) {
            int sms = 0;
            e = sm_count(&sms);
            if (e != cudaSuccess) return e;
            const int64_t want = (int64_t)DETFOLD_FILL_SMS * sms;
            while (threads > 64 && blocks < want) {
                threads /= 2;
                cap *= 2;  // the same resident threads in CTAs of half the size
                per_iter = (int64_t)threads * u;
                blocks = (work + per_iter - 1) / per_iter;
            }
        }
        // every CTA, the extra ones included, resident at once
        if (blocks > cap - extra_blocks) blocks = cap - extra_blocks;
    }
    if (blocks < 1) blocks = 1;
    if (blocks > 0x7FFFFFFF - extra_blocks) blocks = 0x7FFFFFFF - extra_blocks;
    blocks += extra_blocks;  // CTAs with work of their own (a vector kernel's edge CTA)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // the launch attribute follows the kernel's own flag, so a kernel
    // launched early always waits (griddepcontrol.wait) before its loads
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, Kernel, p);
}

// A small-path launch: ceil(work / threads) CTAs of `threads` after
// `extra_blocks` leading CTAs with work of their own (the edge CTA), always
// with programmatic dependent launch when the parameters ask for it.
template <auto Kernel, typename Params>
inline cudaError_t launch_small(const Params &p, int64_t work, int threads, cudaStream_t stream,
                                int extra_blocks = 0)
{
    int64_t blocks = (work + threads - 1) / threads + extra_blocks;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, Kernel, p);
}

template <int NT>
inline FoldParams<NT> fill_params(const LaunchSpec &s, const Plan &pl, bool small)
{
    FoldParams<NT> p = {};
    for (int r = 0; r < s.W; ++r) p.src[r] = s.src[r];
    p.out = s.out;
    p.len = s.len;
    p.head = pl.head;
    p.nvec = pl.nvec;
    p.scale = s.scale;
    p.do_scale = s.do_scale;
    p.W = s.W;
    p.pdl = ((small && DETFOLD_SMALL_PDL) || DETFOLD_PDL_ALL) ? 1 : 0;
    p.edges = (pl.head != 0 || s.len - pl.head - pl.nvec * pl.vec != 0) ? 1 : 0;
    return p;
}

// Bulk-async (TMA) staged bandwidth path (fold_bulk.cu).
int bulk_tile_floats(int W, int mode);  // floats per rank per tile of the bulk path
cudaError_t launch_bulk(const LaunchSpec &s, int64_t head, cudaStream_t stream);
// The bulk-async all-reduce for arenas at different 16-byte phases, W <= 8.
cudaError_t launch_bulk_mixed(const LaunchSpec &s, cudaStream_t stream);
// Large fold or all-reduce over a device-resident pointer table, W <= 8: the
// bulk-async pipeline when the entries share a 16-byte phase (decided on the
// device), else a scalar fold; same status word as the other table kernels.
cudaError_t launch_bulk_table(const float *const *d_table, float *out, int *d_status, int W, int64_t len,
                              float scale, int do_scale, int mode, cudaStream_t stream);
cudaError_t read_pipeline_timeouts_bulk(unsigned long long *count);
cudaError_t read_pipeline_timeouts_move(unsigned long long *count);

template <int W, int MODE>
inline cudaError_t launch_fixed(const LaunchSpec &s, cudaStream_t stream)
{
    const bool small = s.len <= DETFOLD_SMALL_LEN;
    const Plan pl = make_plan(s, small ? DETFOLD_SMALL_VEC : DETFOLD_PREFER_VEC);
    if (DETFOLD_USE_BULK && !small && pl.vec >= 4 && s.len >= DETFOLD_BULK_MIN_LEN &&
        s.len - pl.head >= bulk_tile_floats(W, MODE))
        return launch_bulk(s, pl.head, stream);
    const FoldParams<W> p = fill_params<W>(s, pl, small);
    constexpr int T = bw_threads<MODE>();
    constexpr int C = ctas_per_sm_cap<MODE>();
    if (small && pl.vec != 0) {
        // the fewest vectors take smaller CTAs, spread over more SMs
        const int threads = pl.nvec <= DETFOLD_TINY_VECS ? DETFOLD_TINY_THREADS : DETFOLD_SMALL_THREADS;
        const bool exact = DETFOLD_SMALL_EXACT && pl.nvec > 0 && pl.nvec % threads == 0 && !p.edges;
        const int e = p.edges;  // the edge CTA
        if (pl.vec == 8)
            return exact ? launch_small<fold_small_kernel<W, 8, MODE, true>>(p, pl.nvec, threads, stream, e)
                         : launch_small<fold_small_kernel<W, 8, MODE, false>>(p, pl.nvec, threads, stream, e);
        return exact ? launch_small<fold_small_kernel<W, 4, MODE, true>>(p, pl.nvec, threads, stream, e)
                     : launch_small<fold_small_kernel<W, 4, MODE, false>>(p, pl.nvec, threads, stream, e);
    }
    // a vector kernel whose CTA was shrunk to fit its registers gets as many
    // more CTAs per SM as the cap allows, so the threads per SM stay the same
    if (pl.vec == 8) {
        constexpr int U = u_for<MODE>(W, 8);
        constexpr int VT = vec_threads<W, 8, U, MODE>();
        return launch_kernel<fold_vec_kernel<W, 8, U, MODE>>(p, pl.nvec, U, small, VT, C * (T / VT), stream);
    }
    if (pl.vec == 4) {
        constexpr int U = u_for<MODE>(W, 4);
        constexpr int VT = vec_threads<W, 4, U, MODE>();
        return launch_kernel<fold_vec_kernel<W, 4, U, MODE>>(p, pl.nvec, U, small, VT, C * (T / VT), stream);
    }
    if constexpr (MODE == kAllReduce) {
        // no common 16-byte phase, large: the bulk-async pipeline with
        // per-arena offsets (fold_bulk.cu)
        if (DETFOLD_USE_BULK && DETFOLD_BULK_MIXED && !small && pl.vec == 0 && s.len >= DETFOLD_BULK_MIN_LEN)
            return launch_bulk_mixed(s, stream);
    }
    if (MODE != kAllReduce || DETFOLD_AR_REALIGN) {
        // no common phase: realign every operand onto one 32-byte grid, the
        // output's for a sum, arena 0's for the all-reduce
        RealignParams<W> q = {};
        const int ph = elem_phase(MODE == kAllReduce ? (const void *)s.src[0] : (const void *)s.out, 8);
        q.head = (8 - ph) % 8;
        if (q.head > s.len) q.head = s.len;
        q.nvec = (s.len - q.head) / 8;
        for (int r = 0; r < W; ++r) {
            q.src[r] = s.src[r];
            q.shift[r] = elem_phase(s.src[r] + q.head, 8);
        }
        q.out = s.out;
        q.len = s.len;
        q.scale = s.scale;
        q.do_scale = s.do_scale;
        q.pdl = p.pdl;
        // a warp covers 31 vectors per pass, DETFOLD_REALIGN_U passes per
        // iteration; one warp more, with no pass, folds the scalar edges
        const int64_t work = (q.nvec > 2 ? (q.nvec - 2 + 30) / 31 * 32 : 0) + 32;
        static_assert(DETFOLD_SMALL_THREADS <= DETFOLD_REALIGN_THREADS, "small launches fit the launch bound");
        // (its CTA size stays: smaller CTAs measured slower for this kernel)
        return launch_kernel<fold_realign_kernel<W, MODE>>(q, work, DETFOLD_REALIGN_U, small,
                                                           DETFOLD_REALIGN_THREADS, 0, stream, false);
    }
    constexpr int U = u_for<MODE>(W, 0);
    return launch_kernel<fold_scalar_kernel<W, U, MODE>>(p, s.len, U, small, T, C, stream);
}

template <int MODE>
inline cudaError_t launch_generic(const LaunchSpec &s, cudaStream_t stream)
{
    const bool small = s.len <= DETFOLD_SMALL_LEN;
    const Plan pl = make_plan(s, small ? DETFOLD_SMALL_VEC : DETFOLD_PREFER_VEC);
    const FoldParams<kGenericW> p = fill_params<kGenericW>(s, pl, small);
    constexpr int T = bw_threads<MODE>();
    constexpr int C = ctas_per_sm_cap<MODE>();
    if (pl.vec == 8) return launch_kernel<fold_vec_generic_kernel<8, MODE>>(p, pl.nvec, 1, small, T, C, stream);
    if (pl.vec == 4) return launch_kernel<fold_vec_generic_kernel<4, MODE>>(p, pl.nvec, 1, small, T, C, stream);
    return launch_kernel<fold_scalar_generic_kernel<MODE>>(p, s.len, 1, small, T, C, stream);
}

template <int MODE>
inline cudaError_t launch_mode(const LaunchSpec &s, cudaStream_t stream)
{
    switch (s.W) {
    case 1: return launch_fixed<1, MODE>(s, stream);
    case 2: return launch_fixed<2, MODE>(s, stream);
    case 3: return launch_fixed<3, MODE>(s, stream);
    case 4: return launch_fixed<4, MODE>(s, stream);
    case 5: return launch_fixed<5, MODE>(s, stream);
    case 6: return launch_fixed<6, MODE>(s, stream);
    case 7: return launch_fixed<7, MODE>(s, stream);
    case 8: return launch_fixed<8, MODE>(s, stream);
    default: return launch_generic<MODE>(s, stream);
    }
}

// Defined one per translation unit (fold_sum_nc.cu, fold_sum_coherent.cu,
// fold_allreduce.cu) so the instantiations compile in parallel.
cudaError_t launch_sum_nc(const LaunchSpec &s, cudaStream_t stream);
cudaError_t launch_sum_coherent(const LaunchSpec &s, cudaStream_t stream);
cudaError_t launch_allreduce(const LaunchSpec &s, cudaStream_t stream);
// Fold or all-reduce over a device-resident pointer table (fold_table.cu).
cudaError_t launch_table(const float *const *d_table, float *out, int *d_status, int W, int64_t len,
                         float scale, int do_scale, int mode, cudaStream_t stream);
// Pure movement of K pairs (move_kernels.cu); K may exceed kMaxPairs.
cudaError_t launch_move(const float *const *src, float *const *dst, int K, int64_t len,
                        cudaStream_t stream);

}  // namespace detfold
