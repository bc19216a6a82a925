// Device side of libdetfold: the vector fold kernels for sm_103a.
//
// Every fold of the library computes, per element i, the serial chain
//     acc = s_0[i]; acc = __fadd_rn(acc, s_r[i]) for r = 1..W-1
// in ascending source-rank order (mamba-rs 0.6.2 src/dist/reducer.rs,
// `DET_SUM_RANKS_SRC` and `reduce_sum_reference`), optionally multiplies by
// the mean scale with one __fmul_rn (module doc of the same page), and stores.
// No lane ever combines values of another element, so the bits do not depend
// on the kernel, the grid, the vector width or the unroll depth.
//
// This header holds the load-into-registers kernels:
//   fold_small_kernel     W <= 8, len <= DETFOLD_SMALL_LEN, one phase: one
//                         vector per thread, head and tail in a leading CTA;
//   fold_vec_kernel       W <= 8, every operand at one 32- or 16-byte phase:
//                         scalar head, vector body (all loads of a group
//                         issued before any add), scalar tail;
//   fold_realign_kernel   operands at different 4-byte phases: vectors on
//                         one reference grid, straddles rebuilt with warp
//                         shuffles (the all-reduce also assembles each
//                         arena's aligned stores from two lanes' results);
//   fold_scalar_kernel    the all-reduce at mismatched phases when
//                         DETFOLD_AR_REALIGN is 0;
//   fold_vec/scalar_generic_kernel   8 < W <= 256.
// Large aligned calls, and large all-reduces whose arenas sit at different
// 16-byte phases, take the bulk-async (TMA) kernels of fold_bulk.cu;
// device-resident pointer tables take fold_table.cu.
//
// Modes:
//   kSumNC        out <- fold(src); sources read through the read-only path
//                 (out is disjoint from every source).
//   kSumCoherent  the same with ordinary loads (out may equal one source:
//                 the in-place fold).
//   kAllReduce    every arena <- fold(arenas); ordinary loads, then W stores
//                 (each element is read, then written, by the same thread --
//                 by the same warp in the realigned kernel).
//
// Every launch uses programmatic dependent launch: a kernel executes
// `griddepcontrol.wait` before its first load (its inputs may come from the
// preceding kernel) and `griddepcontrol.launch_dependents` right after, so
// the next grid is resident when this one retires. There are no spin waits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Launch-shape knobs (compile-time; the defaults are the measured choice).
#ifndef DETFOLD_PREFER_VEC
#define DETFOLD_PREFER_VEC 8  // 8 = 32-byte vectors, 4 = 16-byte vectors
#endif
#ifndef DETFOLD_SUM_INFLIGHT
#define DETFOLD_SUM_INFLIGHT 256  // loaded bytes per thread per unrolled group, sum modes
#endif
#ifndef DETFOLD_AR_INFLIGHT
#define DETFOLD_AR_INFLIGHT 256  // the same for the all-reduce mode
#endif
#ifndef DETFOLD_SCALE_INFLIGHT
#define DETFOLD_SCALE_INFLIGHT 512  // the same for the W=1 scale pass (the mean pass)
#endif
#ifndef DETFOLD_SUM_MAX_FLOATS
#define DETFOLD_SUM_MAX_FLOATS 32  // cap on loaded floats per thread per group (U > 1), sum modes
#endif
#ifndef DETFOLD_SCALAR_INFLIGHT
#define DETFOLD_SCALAR_INFLIGHT 32  // the same for the scalar (mismatched-phase) kernels
#endif
#ifndef DETFOLD_SCALAR_MAX_U
#define DETFOLD_SCALAR_MAX_U 16
#endif
#ifndef DETFOLD_SMALL_LEN
#define DETFOLD_SMALL_LEN (1 << 17)  // elements at or below: small-payload launch
#endif
#ifndef DETFOLD_SMALL_VEC
#define DETFOLD_SMALL_VEC DETFOLD_PREFER_VEC  // widest vector on the small path
#endif
#ifndef DETFOLD_SMALL_EXACT
#define DETFOLD_SMALL_EXACT 1  // small-path kernel without the bounds test when the grid is exact
#endif
#ifndef DETFOLD_TINY_VECS
#define DETFOLD_TINY_VECS 0  // small-path calls of at most this many vectors use DETFOLD_TINY_THREADS
#endif
#ifndef DETFOLD_TINY_THREADS
#define DETFOLD_TINY_THREADS 32
#endif
#ifndef DETFOLD_SMALL_THREADS
#define DETFOLD_SMALL_THREADS 128
#endif
#ifndef DETFOLD_SUM_THREADS
#define DETFOLD_SUM_THREADS 1024  // CTA size of the bandwidth path, sum modes
#endif
#ifndef DETFOLD_AR_THREADS
#define DETFOLD_AR_THREADS 256  // CTA size of the bandwidth path, all-reduce mode
#endif
#ifndef DETFOLD_USE_BULK
#define DETFOLD_USE_BULK 1  // bulk-async (TMA) staged path for large aligned calls
#endif
#ifndef DETFOLD_BULK_MIXED
#define DETFOLD_BULK_MIXED 1  // large all-reduce at mixed 16-byte phases: the bulk-async pipeline
#endif
#ifndef DETFOLD_AR_REALIGN
#define DETFOLD_AR_REALIGN 1  // all-reduce at mismatched phases: realigned vectors (0: scalar kernel)
#endif
#ifndef DETFOLD_REALIGN_THREADS
#define DETFOLD_REALIGN_THREADS 256  // CTA size of the realigned kernel
#endif
#ifndef DETFOLD_REALIGN_U
#define DETFOLD_REALIGN_U 1  // warp passes per iteration of the realigned kernel (loads issued together)
#endif
#ifndef DETFOLD_REALIGN_AR_NOALLOC
#define DETFOLD_REALIGN_AR_NOALLOC 0  // 1: the realigned kernel's coherent loads skip L1
#endif
#ifndef DETFOLD_USE_BULK_MOVE
#define DETFOLD_USE_BULK_MOVE 1  // bulk-async path for large pure-movement launches
#endif
#ifndef DETFOLD_BULK_MIN_LEN
#define DETFOLD_BULK_MIN_LEN (1 << 21)  // elements at or above: the bulk path (folds, parameter table)
#endif
#ifndef DETFOLD_BULK_TABLE_MIN_LEN
#define DETFOLD_BULK_TABLE_MIN_LEN (1 << 20)  // the same for folds over a device-resident table
#endif
#ifndef DETFOLD_BULK_MOVE_MIN_LEN
#define DETFOLD_BULK_MOVE_MIN_LEN (1 << 20)  // the same for pure-movement launches
#endif
#ifndef DETFOLD_SMALL_PDL
#define DETFOLD_SMALL_PDL 1  // programmatic dependent launch on the small path
#endif
#ifndef DETFOLD_PDL_ALL
#define DETFOLD_PDL_ALL 1  // ... and on every other launch (0 restricts it to the small path)
#endif
#ifndef DETFOLD_PDL_TRIGGER_FIRST
#define DETFOLD_PDL_TRIGGER_FIRST 0  // 1: launch_dependents before the wait instead of after
#endif
#ifndef DETFOLD_SUM_CTAS_PER_SM
#define DETFOLD_SUM_CTAS_PER_SM 1  // 0: as many as fit; else at most this many per SM
#endif
#ifndef DETFOLD_AR_CTAS_PER_SM
#define DETFOLD_AR_CTAS_PER_SM 0
#endif
#ifndef DETFOLD_FILL_SMS
#define DETFOLD_FILL_SMS 2  // bandwidth-path grids below this many CTAs per SM use smaller CTAs (0: off)
#endif

// Cache-hint knobs (compile-time; the defaults are the measured choice).
#ifndef DETFOLD_LD_L2_PREFETCH
#define DETFOLD_LD_L2_PREFETCH 0  // 0, 128 or 256: L2 prefetch size hint on vector loads
#endif
#ifndef DETFOLD_ST_HINT
#define DETFOLD_ST_HINT 0  // 0: default write-back, 1: .cs (streaming), 2: .L1::no_allocate
#endif
#if DETFOLD_LD_L2_PREFETCH == 256
#define DETFOLD_LD_PF ".L2::256B"
#elif DETFOLD_LD_L2_PREFETCH == 128
#define DETFOLD_LD_PF ".L2::128B"
#else
#define DETFOLD_LD_PF ""
#endif
#if DETFOLD_ST_HINT == 1
#define DETFOLD_ST_Q ".cs"
#elif DETFOLD_ST_HINT == 2
#define DETFOLD_ST_Q ".L1::no_allocate"
#else
#define DETFOLD_ST_Q ""
#endif

namespace detfold {

enum Mode : int { kSumNC = 0, kSumCoherent = 1, kAllReduce = 2 };

// CTA size of the bandwidth path, and the launch bound that also admits the
// small path's CTAs.
template <int MODE>
constexpr int bw_threads()
{
    return MODE == kAllReduce ? DETFOLD_AR_THREADS : DETFOLD_SUM_THREADS;
}
template <int MODE>
constexpr int ctas_per_sm_cap()
{
    return MODE == kAllReduce ? DETFOLD_AR_CTAS_PER_SM : DETFOLD_SUM_CTAS_PER_SM;
}
template <int MODE>
constexpr int max_threads()
{
    return bw_threads<MODE>() > DETFOLD_SMALL_THREADS ? bw_threads<MODE>() : DETFOLD_SMALL_THREADS;
}

// CTA size of the vector kernel: the mode's size, halved while a thread's
// live values -- W*VEC*U loaded floats, W*U 64-bit addresses and about 24
// registers of indices and loop state -- would exceed the registers that size
// leaves per thread (65536 / threads), so no instantiation spills.
template <int W, int VEC, int U, int MODE>
constexpr int vec_threads()
{
    int t = bw_threads<MODE>();
    while (t > 128 && W * VEC * U + 2 * W * U + 24 > 65536 / t) t /= 2;
    return t;
}

constexpr int kGenericW = 256;  // table capacity of the runtime-W kernels

template <int NT>
struct FoldParams {
    const float *src[NT];  // sources (kAllReduce: the arenas, also written)
    float *out;            // destination of the sum modes
    int64_t len;           // elements
    int64_t head;          // scalar elements before the vector body
    int64_t nvec;          // vectors in the body
    float scale;           // applied when do_scale != 0
    int do_scale;
    int W;                 // runtime world size (used by the generic kernels)
    int pdl;               // launched with programmatic dependent launch
    int edges;             // the call has a head or a tail (small-payload kernel: edge CTA)
};

// Pure-movement launches: K (source -> destination) pairs of equal length.
// 250 pairs keep the parameter block under 4 KB; longer lists are split.
constexpr int kMaxPairs = 250;
struct MoveParams {
    const float *src[kMaxPairs];
    float *dst[kMaxPairs];
    int64_t len, head, nvec;
    int K;
    short pdl;
    short edge_blocks;  // leading CTAs that move only the head and tail elements (at most 28)
};
static_assert(sizeof(MoveParams) == 2 * kMaxPairs * sizeof(void *) + 32, "the parameter block stays 4032 bytes");

template <int VEC>
struct alignas(VEC * 4) Vec {
    float v[VEC];
};

// ---------------------------------------------------------------- loads / stores

template <bool NC>
__device__ __forceinline__ float ld1(const float *p)
{
    float x;
    if constexpr (NC)
        asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(x) : "l"(p));
    else
        asm volatile("ld.global.L1::no_allocate.f32 %0, [%1];" : "=f"(x) : "l"(p));
    return x;
}

template <int VEC, bool NC>
__device__ __forceinline__ Vec<VEC> ldv(const float *p)
{
    Vec<VEC> r;
    if constexpr (VEC == 4) {
        if constexpr (NC)
            asm volatile("ld.global.nc.L1::no_allocate" DETFOLD_LD_PF ".v4.f32 {%0,%1,%2,%3}, [%4];"
                : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3])
                : "l"(p));
        else
            asm volatile("ld.global.L1::no_allocate" DETFOLD_LD_PF ".v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3])
                         : "l"(p));
    } else {
        static_assert(VEC == 8, "VEC is 4 or 8");
        if constexpr (NC)
            asm volatile("ld.global.nc.L1::no_allocate" DETFOLD_LD_PF ".v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                  "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                : "l"(p));
        else
            asm volatile("ld.global.L1::no_allocate" DETFOLD_LD_PF ".v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]),
                           "=f"(r.v[4]), "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                         : "l"(p));
    }
    return r;
}

__device__ __forceinline__ void st1(float *p, float x)
{
    asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(x) : "memory");
}

template <int VEC>
__device__ __forceinline__ void stv(float *p, const Vec<VEC> &x)
{
    if constexpr (VEC == 4)
        asm volatile("st.global" DETFOLD_ST_Q ".v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(x.v[0]), "f"(x.v[1]),
                     "f"(x.v[2]), "f"(x.v[3])
                     : "memory");
    else
        asm volatile("st.global" DETFOLD_ST_Q ".v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(x.v[0]),
                     "f"(x.v[1]), "f"(x.v[2]), "f"(x.v[3]), "f"(x.v[4]), "f"(x.v[5]),
                     "f"(x.v[6]), "f"(x.v[7])
                     : "memory");
}

// Either order is correct: launch_dependents only lets the next grid be
// scheduled; that grid's own wait still blocks until this grid has retired
// and its writes are visible.
__device__ __forceinline__ void pdl_enter(int pdl)
{
    if (pdl) {
#if DETFOLD_PDL_TRIGGER_FIRST
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
#else
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    }
}

// ---------------------------------------------------------------- one element

// The full chain for element i with scalar accesses (head, tail, scalar path).
template <int W, int MODE, int NT>
__device__ __forceinline__ void fold_one(const FoldParams<NT> &p, int64_t i)
{
    constexpr bool NC = (MODE == kSumNC);
    const int w = (W > 0) ? W : p.W;
    float acc = ld1<NC>(p.src[0] + i);
    if constexpr (W > 0) {
#pragma unroll
        for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, ld1<NC>(p.src[r] + i));
    } else {
        for (int r = 1; r < w; ++r) acc = __fadd_rn(acc, ld1<NC>(p.src[r] + i));
    }
    if (p.do_scale) acc = __fmul_rn(acc, p.scale);
    if constexpr (MODE == kAllReduce) {
        for (int r = 0; r < w; ++r) st1(const_cast<float *>(p.src[r]) + i, acc);
    } else {
        st1(p.out + i, acc);
    }
}

template <int VEC, int W, int MODE, int NT>
__device__ __forceinline__ void store_result(const FoldParams<NT> &p, int64_t e, Vec<VEC> acc)
{
    if (p.do_scale) {
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc.v[k] = __fmul_rn(acc.v[k], p.scale);
    }
    if constexpr (MODE == kAllReduce) {
        const int w = (W > 0) ? W : p.W;
        if constexpr (W > 0) {
#pragma unroll
            for (int r = 0; r < W; ++r) stv<VEC>(const_cast<float *>(p.src[r]) + e, acc);
        } else {
            for (int r = 0; r < w; ++r) stv<VEC>(const_cast<float *>(p.src[r]) + e, acc);
        }
    } else {
        stv<VEC>(p.out + e, acc);
    }
}

// ---------------------------------------------------------------- vector kernel, fixed W

// U vectors per thread per iteration, grid-stride; every operand shares the
// same VEC*4-byte phase. Element index of vector v is head + v*VEC.
template <int W, int VEC, int U, int MODE>
__global__ void __launch_bounds__(vec_threads<W, VEC, U, MODE>()) fold_vec_kernel(const __grid_constant__ FoldParams<W> p)
{
    constexpr bool NC = (MODE == kSumNC);
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t v = gtid;
    for (; v + (U - 1) * stride < p.nvec; v += U * stride) {
        Vec<VEC> x[U][W];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < W; ++r)
                x[u][r] = ldv<VEC, NC>(p.src[r] + p.head + (v + u * stride) * VEC);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            Vec<VEC> acc = x[u][0];
#pragma unroll
            for (int r = 1; r < W; ++r)
#pragma unroll
                for (int k = 0; k < VEC; ++k) acc.v[k] = __fadd_rn(acc.v[k], x[u][r].v[k]);
            store_result<VEC, W, MODE>(p, p.head + (v + u * stride) * VEC, acc);
        }
    }
    for (; v < p.nvec; v += stride) {
        Vec<VEC> x[W];
#pragma unroll
        for (int r = 0; r < W; ++r) x[r] = ldv<VEC, NC>(p.src[r] + p.head + v * VEC);
        Vec<VEC> acc = x[0];
#pragma unroll
        for (int r = 1; r < W; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc.v[k] = __fadd_rn(acc.v[k], x[r].v[k]);
        store_result<VEC, W, MODE>(p, p.head + v * VEC, acc);
    }
    // head and tail: fewer than VEC elements each
    const int64_t tail0 = p.head + p.nvec * VEC;
    if (gtid < p.head) fold_one<W, MODE>(p, gtid);
    if (gtid < p.len - tail0) fold_one<W, MODE>(p, tail0 + gtid);
}

// ---------------------------------------------------------------- small-payload kernel, fixed W

// The head and the tail of a small call (fewer than VEC elements each):
// thread i < VEC of the edge CTA folds head element i, thread VEC + j tail
// element j, so no thread has two round trips. Inline: an out-of-line call
// measured about 0.4 us more per 16 KiB call than the vectors' own round trip.
template <int W, int VEC, int MODE>
__device__ __forceinline__ void fold_edges(const FoldParams<W> &p, int i)
{
    const int head = (int)p.head, tail0 = head + (int)p.nvec * VEC;
    if (i < VEC ? i < head : i - VEC < (int)p.len - tail0)
        fold_one<W, MODE>(p, i < VEC ? i : tail0 + (i - VEC));
}

// The small path (len <= DETFOLD_SMALL_LEN), every operand at one phase: one
// vector per thread, no loop, 32-bit indices. Back to back in a graph, such
// a launch costs about what its CTAs execute after the wait, so the body is
// only the W loads, the chain and the store. EXACT: a call with no edges
// whose CTAs have exactly one thread per vector (nvec a multiple of the CTA
// size), so no bounds test and no edge CTA.
static_assert(DETFOLD_TINY_THREADS >= 16 && DETFOLD_SMALL_THREADS >= 16, "an edge CTA has a thread per edge element");

template <int W, int VEC, int MODE, bool EXACT>
__global__ void __launch_bounds__(DETFOLD_SMALL_THREADS) fold_small_kernel(const __grid_constant__ FoldParams<W> p)
{
    static_assert(DETFOLD_SMALL_LEN < (1 << 30), "small-path indices are 32-bit");
    constexpr bool NC = (MODE == kSumNC);
    pdl_enter(p.pdl);
    // a call with edges (never an EXACT one) has one more CTA, the first, for
    // them alone, so no thread adds their round trip to its vector's
    int b = blockIdx.x;
    if constexpr (!EXACT) {
        if (p.edges) {
            if (b == 0) {
                if (threadIdx.x < 2 * VEC) fold_edges<W, VEC, MODE>(p, threadIdx.x);
                return;
            }
            b -= 1;
        }
    }
    const int i = b * blockDim.x + threadIdx.x;
    if (EXACT || i < (int)p.nvec) {
        const int e = (int)p.head + i * VEC;
        Vec<VEC> x[W];
#pragma unroll
        for (int r = 0; r < W; ++r) x[r] = ldv<VEC, NC>(p.src[r] + e);
        Vec<VEC> acc = x[0];
#pragma unroll
        for (int r = 1; r < W; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc.v[k] = __fadd_rn(acc.v[k], x[r].v[k]);
        store_result<VEC, W, MODE>(p, e, acc);
    }
}

// ---------------------------------------------------------------- scalar kernel, fixed W

// Operands at different 4-byte phases: coalesced scalar accesses, U elements
// per thread per iteration with all U*W loads issued first.
template <int W, int U, int MODE>
__global__ void __launch_bounds__(max_threads<MODE>()) fold_scalar_kernel(const __grid_constant__ FoldParams<W> p)
{
    constexpr bool NC = (MODE == kSumNC);
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (U - 1) * stride < p.len; i += U * stride) {
        float x[U][W];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < W; ++r) x[u][r] = ld1<NC>(p.src[r] + i + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float acc = x[u][0];
#pragma unroll
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, x[u][r]);
            if (p.do_scale) acc = __fmul_rn(acc, p.scale);
            if constexpr (MODE == kAllReduce) {
#pragma unroll
                for (int r = 0; r < W; ++r) st1(const_cast<float *>(p.src[r]) + i + u * stride, acc);
            } else {
                st1(p.out + i + u * stride, acc);
            }
        }
    }
    for (; i < p.len; i += stride) fold_one<W, MODE>(p, i);
}

// ---------------------------------------------------------------- runtime-W kernels (W > 8)

// Loads are issued G ranks at a time ahead of their adds (G*VEC*4 = 128
// bytes per thread); the chain order is unchanged.
template <int VEC, int MODE>
__global__ void __launch_bounds__(max_threads<MODE>()) fold_vec_generic_kernel(const __grid_constant__ FoldParams<kGenericW> p)
{
    constexpr bool NC = (MODE == kSumNC);
    constexpr int G = 32 / VEC;
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t v = gtid; v < p.nvec; v += stride) {
        const int64_t e = p.head + v * VEC;
        Vec<VEC> acc = ldv<VEC, NC>(p.src[0] + e);
        for (int r0 = 1; r0 < p.W; r0 += G) {
            Vec<VEC> x[G];
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (r0 + k < p.W) x[k] = ldv<VEC, NC>(p.src[r0 + k] + e);
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (r0 + k < p.W)
#pragma unroll
                    for (int j = 0; j < VEC; ++j) acc.v[j] = __fadd_rn(acc.v[j], x[k].v[j]);
        }
        store_result<VEC, 0, MODE>(p, e, acc);
    }
    const int64_t tail0 = p.head + p.nvec * VEC;
    if (gtid < p.head) fold_one<0, MODE>(p, gtid);
    if (gtid < p.len - tail0) fold_one<0, MODE>(p, tail0 + gtid);
}

template <int MODE>
__global__ void __launch_bounds__(max_threads<MODE>()) fold_scalar_generic_kernel(const __grid_constant__ FoldParams<kGenericW> p)
{
    constexpr bool NC = (MODE == kSumNC);
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.len; i += stride) {
        float acc = ld1<NC>(p.src[0] + i);
        for (int r0 = 1; r0 < p.W; r0 += 8) {
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < p.W) x[k] = ld1<NC>(p.src[r0 + k] + i);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < p.W) acc = __fadd_rn(acc, x[k]);
        }
        if (p.do_scale) acc = __fmul_rn(acc, p.scale);
        if constexpr (MODE == kAllReduce) {
            for (int r = 0; r < p.W; ++r) st1(const_cast<float *>(p.src[r]) + i, acc);
        } else {
            st1(p.out + i, acc);
        }
    }
}

// ---------------------------------------------------------------- realigned vector kernel

// Operands at different 4-byte phases (e.g. the rows of a [W][len] stack
// when len % 8 != 0, or arenas at per-rank offsets). Logical vectors of 8
// elements follow one reference 32-byte grid: the output's for the sums,
// arena 0's for the all-reduce. Operand r's eight elements of logical vector
// v straddle two of its aligned 32-byte vectors, at element shift d_r =
// phase of (src_r + head). Each lane loads one aligned vector per operand;
// the upper half of its straddle is the next lane's vector, taken with a
// warp shuffle. A warp therefore folds 31 logical vectors per pass: lane 31
// only loads, to feed lane 30. The body covers logical vectors 1 .. nvec-2
// (loads 1 .. nvec-1), which keeps every load inside every operand; the
// edges are scalar.
//
// The all-reduce stores the mirror image: the aligned vector a lane loaded
// from arena r holds the last d_r elements of logical vector v-1 (folded by
// the previous lane, taken with an upward shuffle) and the first 8-d_r of
// v (its own). A lane stores it whole when the pass folded both; at a pass's
// two ends it stores only the elements the pass folded, one by one. So every
// element is written once, by the pass that folded it, and a pass uses only
// elements that no other pass writes: the other elements of the vectors it
// loads at its ends are loaded but never used, and the update in place needs
// no ordering between passes.
template <int NT>
struct RealignParams {
    const float *src[NT];
    int shift[NT];  // d_r in 0..7
    float *out;
    int64_t len, head, nvec;
    float scale;
    int do_scale;
    int pdl;
};

// Realigned kernel loads. They allocate in L1 (the vector at a pass's end
// is loaded again by the next pass), except in the coherent modes (in-place
// fold, all-reduce) when DETFOLD_REALIGN_AR_NOALLOC is set. NC: the
// read-only path.
template <bool NC>
__device__ __forceinline__ Vec<8> ldv8_l1(const float *p)
{
    Vec<8> r;
    if constexpr (!NC && DETFOLD_REALIGN_AR_NOALLOC)
        return ldv<8, false>(p);
    if constexpr (NC)
        asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                       "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                     : "l"(p));
    else
        asm volatile("ld.global.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                       "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                     : "l"(p));
    return r;
}

template <int D>
__device__ __forceinline__ Vec<8> take8(const Vec<8> &a, const Vec<8> &b)
{
    Vec<8> x;
#pragma unroll
    for (int k = 0; k < 8; ++k) x.v[k] = (k + D < 8) ? a.v[k + D] : b.v[k + D - 8];
    return x;
}

// x[k] = a[k+D] for k+D < 8, else b[k+D-8], for a warp-uniform runtime D in 0..7.
__device__ __forceinline__ Vec<8> take8_rt(const Vec<8> &a, const Vec<8> &b, int d)
{
    switch (d) {
    case 0: return a;
    case 1: return take8<1>(a, b);
    case 2: return take8<2>(a, b);
    case 3: return take8<3>(a, b);
    case 4: return take8<4>(a, b);
    case 5: return take8<5>(a, b);
    case 6: return take8<6>(a, b);
    default: return take8<7>(a, b);
    }
}

// One pass of a warp over logical vectors v = 1 + 31c + lane, with the
// lane's aligned vectors of every operand already loaded into lo[].
template <int W, int MODE>
__device__ __forceinline__ void realign_pass(const RealignParams<W> &p, const Vec<8> (&lo)[W], int64_t v,
                                             int lane)
{
    const bool writes = lane < 31 && v <= p.nvec - 2;
    const int64_t e = p.head + v * 8;
    Vec<8> acc;
#pragma unroll
    for (int r = 0; r < W; ++r) {
        Vec<8> x;
        const int d = p.shift[r];  // uniform: no divergence
        if (d == 0) {
            x = lo[r];
        } else {
            Vec<8> hi;
#pragma unroll
            for (int k = 0; k < 8; ++k) hi.v[k] = __shfl_down_sync(0xffffffffu, lo[r].v[k], 1);
            x = take8_rt(lo[r], hi, d);
        }
        if (r == 0) {
            acc = x;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc.v[k] = __fadd_rn(acc.v[k], x.v[k]);
        }
    }
    if (p.do_scale) {
#pragma unroll
        for (int k = 0; k < 8; ++k) acc.v[k] = __fmul_rn(acc.v[k], p.scale);
    }
    if constexpr (MODE == kAllReduce) {
        // the previous lane's result: the head of every arena's aligned
        // vector at this lane
        Vec<8> prev;
#pragma unroll
        for (int k = 0; k < 8; ++k) prev.v[k] = __shfl_up_sync(0xffffffffu, acc.v[k], 1);
        const bool own_prev = lane > 0 && v - 1 <= p.nvec - 2;  // logical v-1 folded in this pass
        const bool own_cur = writes;                            // logical v folded in this pass
#pragma unroll
        for (int r = 0; r < W; ++r) {
            const int d = p.shift[r];
            float *dst = const_cast<float *>(p.src[r]) + e - d;  // the aligned vector loaded
            if (d == 0) {
                if (own_cur) stv<8>(dst, acc);
            } else if (own_prev || own_cur) {
                const Vec<8> x = take8_rt(prev, acc, 8 - d);  // x[m] = prev[8-d+m] (m < d), acc[m-d]
                if (own_prev && own_cur) {
                    stv<8>(dst, x);
                } else {
#pragma unroll
                    for (int m = 0; m < 8; ++m)
                        if (m < d ? own_prev : own_cur) st1(dst + m, x.v[m]);
                }
            }
        }
    } else if (writes) {
        stv<8>(p.out + e, acc);
    }
}

// A warp runs DETFOLD_REALIGN_U passes per iteration (passes c, c + nwarps,
// ...), with the loads of all of them issued before the first pass's
// shuffles, so more bytes are in flight per thread.
template <int W, int MODE>
__global__ void __launch_bounds__(DETFOLD_REALIGN_THREADS) fold_realign_kernel(const __grid_constant__ RealignParams<W> p)
{
    constexpr bool NC = (MODE == kSumNC);
    constexpr int U = DETFOLD_REALIGN_U;
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = stride >> 5;
    // warp-uniform loop: every lane of a warp runs every pass (for the shuffles)
    for (int64_t c = gtid >> 5; 1 + c * 31 < p.nvec - 1; c += U * nwarps) {
        Vec<8> lo[U][W];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = 1 + (c + u * nwarps) * 31 + lane;
#pragma unroll
            for (int r = 0; r < W; ++r) {
                if (v <= p.nvec - 1) {
                    lo[u][r] = ldv8_l1<NC>(p.src[r] + p.head + v * 8 - p.shift[r]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) lo[u][r].v[k] = 0.0f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) realign_pass<W, MODE>(p, lo[u], 1 + (c + u * nwarps) * 31 + lane, lane);
    }
    // scalar edges: [0, lo_end) and [hi_begin, len), disjoint from the body
    // and from each other, taken by the grid's last threads: the host sizes
    // a one-wave grid one warp past the passes, so that warp has no pass and
    // folds the edges beside the body instead of after a pass. No body store
    // covers an edge element. The first and last passes do load the aligned
    // vectors that straddle an edge, but use none of their edge elements, so
    // an edge store landing before those loads changes no result.
    const int64_t body = p.nvec >= 3 ? p.nvec - 2 : 0;
    const int64_t lo_end = body ? p.head + 8 : p.len;
    const int64_t hi_begin = body ? p.head + 8 * (p.nvec - 1) : p.len;
    const int64_t etid = stride - 1 - gtid;
    for (int part = 0; part < 2; ++part) {
        for (int64_t i = (part ? hi_begin : 0) + etid; i < (part ? p.len : lo_end); i += stride) {
            float acc = ld1<NC>(p.src[0] + i);
#pragma unroll
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, ld1<NC>(p.src[r] + i));
            if (p.do_scale) acc = __fmul_rn(acc, p.scale);
            if constexpr (MODE == kAllReduce) {
#pragma unroll
                for (int r = 0; r < W; ++r) st1(const_cast<float *>(p.src[r]) + i, acc);
            } else {
                st1(p.out + i, acc);
            }
        }
    }
}

}  // namespace detfold
