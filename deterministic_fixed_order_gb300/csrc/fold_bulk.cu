// Bandwidth path with bulk-async (TMA) staging: the fold and the fused
// all-reduce for large aligned calls, and the all-reduce for large calls
// whose arenas sit at different 16-byte phases (fold_bulk_mixed_kernel).
//
// Per CTA, one producer lane streams tiles of every rank's operand into a
// ring of shared-memory stages with cp.async.bulk (global -> shared,
// completion on an mbarrier with a byte count); consumer warps fold the
// stage in ascending rank order with __fadd_rn (the same per-element chain
// as every other fold here, so the same bits: mamba-rs 0.6.2
// src/dist/reducer.rs, `reduce_sum_reference`), apply the mean multiply,
// write the result tile to shared memory, and one consumer thread bulk-stores
// it (shared -> global) to the output -- or to all W arenas for the
// all-reduce, so the result is read from shared memory W times instead of
// being recomputed or reloaded. DRAM sees long contiguous requests (one tile
// per rank and stage) and the SMs issue a handful of instructions per tile.
//
// Every mbarrier wait is bounded (%globaltimer, about one second, and a poll
// cap). On expiry the kernel counts the event in a device counter that
// detfold_pipeline_timeouts() reads, waits (bounded) for its own copies in
// flight, and stops; the call's output is then incomplete and the counter
// says so. The consumer warps meet at a named barrier after every wait and
// vote on its outcome (bar.red.or), so they leave together: the second
// barrier of a tile is reached only by consumers that all passed the first.
//
// Preconditions, checked by the dispatcher: W <= 8, every operand at the same
// 16-byte phase (tiles then start 16-byte aligned), at least one whole tile.
// The head before the first tile (scalar) and the tail after the last (16-byte
// vectors spread over the CTAs that hold the fewest tiles) are folded in the
// same launch.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold.h"
#include "detfold_async.cuh"
#include "detfold_launch.cuh"

namespace detfold {

namespace {

// Tile shapes from GB300 sweeps: 4 KB per rank and 4 stages up to W = 4,
// 4 KB per rank and 2 stages above; four consumer warps. The all-reduce has
// its own shapes (below).
#ifndef DETFOLD_BULK_T_LO
#define DETFOLD_BULK_T_LO 1024  // floats per rank per tile, W <= 4
#endif
#ifndef DETFOLD_BULK_S_LO
#define DETFOLD_BULK_S_LO 4     // stages, W <= 4
#endif
#ifndef DETFOLD_BULK_T_HI
#define DETFOLD_BULK_T_HI 1024  // floats per rank per tile, W > 4
#endif
#ifndef DETFOLD_BULK_S_HI
#define DETFOLD_BULK_S_HI 2     // stages, W > 4
#endif
#ifndef DETFOLD_BULK_NCW
#define DETFOLD_BULK_NCW 4      // consumer warps
#endif
#ifndef DETFOLD_BULK_CTAS_PER_SM
#define DETFOLD_BULK_CTAS_PER_SM 2  // 0: as many as shared memory allows
#endif
// The all-reduce's own shape (it reads and writes W tiles per stage; the sums
// read W and write one), by default the same as the sums'.
#ifndef DETFOLD_BULK_AR_T_LO
#define DETFOLD_BULK_AR_T_LO DETFOLD_BULK_T_LO
#endif
#ifndef DETFOLD_BULK_AR_S_LO
#define DETFOLD_BULK_AR_S_LO DETFOLD_BULK_S_LO
#endif
#ifndef DETFOLD_BULK_AR_T_HI
#define DETFOLD_BULK_AR_T_HI DETFOLD_BULK_T_HI
#endif
#ifndef DETFOLD_BULK_AR_S_HI
#define DETFOLD_BULK_AR_S_HI DETFOLD_BULK_S_HI
#endif
#ifndef DETFOLD_BULK_AR_CTAS_PER_SM
#define DETFOLD_BULK_AR_CTAS_PER_SM DETFOLD_BULK_CTAS_PER_SM
#endif
#ifndef DETFOLD_BULK_AR_PER_W
#define DETFOLD_BULK_AR_PER_W 1  // 1: the all-reduce's shape per W from ArShape; 0: the knobs above
#endif
// All-reduce shapes per W (floats per rank per tile, stages, CTAs per SM),
// from an interleaved A/B sweep on GB300 against the sums' shapes (same
// bits): W=2 +5%, W=3 +3%, W=4 +2-3% (the 4 x 1e8 call 6.47 -> 6.61 TB/s),
// W=8 +6%. W=5-6 measured faster with the sums' shapes and keep them; W=1
// has its own (below).
// The W=1 all-reduce (a scale pass) takes the W=1 sum's deep shape below:
// 6.81 TB/s at 1 GiB against 6.62 with 8 KB tiles in 3 stages at 2 CTAs per SM.
#ifndef DETFOLD_BULK_AR_W1_T
#define DETFOLD_BULK_AR_W1_T 4096  // floats per tile,
#endif
#ifndef DETFOLD_BULK_AR_W1_S
#define DETFOLD_BULK_AR_W1_S 4     // stages,
#endif
#ifndef DETFOLD_BULK_AR_W1_C
#define DETFOLD_BULK_AR_W1_C 1     // CTAs per SM
#endif
template <int W>
struct ArShape {
    static constexpr int T = W == 1 ? DETFOLD_BULK_AR_W1_T : W <= 3 ? 1024 : W == 4 ? 512 : W <= 6 ? 1024 : 256;
    static constexpr int S = W == 1 ? DETFOLD_BULK_AR_W1_S : W <= 3 ? 2 : W == 4 ? 3 : W <= 6 ? 2 : 3;
    static constexpr int C = W == 1 ? DETFOLD_BULK_AR_W1_C : W <= 3 ? 3 : 2;
};
// The W=1 sum (a 1:1 stream) keeps more bytes in flight than the other sums:
// 16 KB tiles in 4 stages (one CTA per SM) measured 6.83 TB/s at 1 GiB
// against 5.84 with the shared 4 KB shape, and 6.60 for a torch device copy.
#ifndef DETFOLD_BULK_SUM_W1_T
#define DETFOLD_BULK_SUM_W1_T 4096
#endif
#ifndef DETFOLD_BULK_SUM_W1_S
#define DETFOLD_BULK_SUM_W1_S 4
#endif
template <int W, int MODE>
struct BulkShape {
    static constexpr bool AR = (MODE == kAllReduce);
    static constexpr bool PER_W = AR && DETFOLD_BULK_AR_PER_W;
    static constexpr int T = PER_W ? ArShape<W>::T
                           : (!AR && W == 1) ? DETFOLD_BULK_SUM_W1_T
                           : W <= 4 ? (AR ? DETFOLD_BULK_AR_T_LO : DETFOLD_BULK_T_LO)
                                    : (AR ? DETFOLD_BULK_AR_T_HI : DETFOLD_BULK_T_HI);
    static constexpr int S = PER_W ? ArShape<W>::S
                           : (!AR && W == 1) ? DETFOLD_BULK_SUM_W1_S
                           : W <= 4 ? (AR ? DETFOLD_BULK_AR_S_LO : DETFOLD_BULK_S_LO)
                                    : (AR ? DETFOLD_BULK_AR_S_HI : DETFOLD_BULK_S_HI);
    static constexpr int CTAS_PER_SM = PER_W ? ArShape<W>::C
                                     : (AR ? DETFOLD_BULK_AR_CTAS_PER_SM : DETFOLD_BULK_CTAS_PER_SM);
    static constexpr int NCW = DETFOLD_BULK_NCW;
    static constexpr int THREADS = 32 * (1 + NCW);
    static constexpr size_t SMEM = (size_t)S * (W + 1) * T * 4 + 2 * S * 8;
    static_assert(T % 4 == 0, "tiles are whole 16-byte vectors (bulk copies move multiples of 16 bytes)");
};

template <int W>
struct BulkParams {
    float *a[W];   // sources (all-reduce: also the destinations)
    float *out;    // sum destination
    int64_t len, head, ntiles;
    float scale;
    int do_scale;
    int pdl;
};

// The elements outside the whole tiles: the head [0, head), fewer than 8, and
// the tail [head + ntiles*T, len), fewer than T. The tail starts where a tile
// would, 16-byte aligned: its whole 16-byte vectors go one per consumer
// thread, starting from the last CTA (the CTAs at the end hold the fewest
// tiles); the head and the tail's last few (fewer than 4) elements are
// scalar, in the last CTA. Consumers do this before their tiles, while the
// producer's first loads are in flight.
template <int W, int MODE>
__device__ __forceinline__ void bulk_edges(const BulkParams<W> &p, int tc)
{
    constexpr int T = BulkShape<W, MODE>::T, NC = 32 * BulkShape<W, MODE>::NCW;
    const int64_t tail0 = p.head + p.ntiles * T;
    const int64_t nv = (p.len - tail0) / 4;
    for (int64_t v = (int64_t)(gridDim.x - 1 - blockIdx.x) * NC + tc; v < nv; v += (int64_t)gridDim.x * NC) {
        const int64_t e = tail0 + v * 4;
        Vec<4> x[W];
#pragma unroll
        for (int r = 0; r < W; ++r) x[r] = ldv<4, false>(p.a[r] + e);
        Vec<4> acc = x[0];
#pragma unroll
        for (int r = 1; r < W; ++r)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc.v[k] = __fadd_rn(acc.v[k], x[r].v[k]);
        if (p.do_scale) {
#pragma unroll
            for (int k = 0; k < 4; ++k) acc.v[k] = __fmul_rn(acc.v[k], p.scale);
        }
        if constexpr (MODE == kAllReduce) {
#pragma unroll
            for (int r = 0; r < W; ++r) stv<4>(p.a[r] + e, acc);
        } else {
            stv<4>(p.out + e, acc);
        }
    }
    if (blockIdx.x != gridDim.x - 1) return;
    const int64_t rest0 = tail0 + nv * 4;
    const int nhead = (int)p.head, nrest = (int)(p.len - rest0);
    if (tc < nhead + nrest) {
        const int64_t i = tc < nhead ? tc : rest0 + (tc - nhead);
        float acc = ld1<false>(p.a[0] + i);
#pragma unroll
        for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, ld1<false>(p.a[r] + i));
        if (p.do_scale) acc = __fmul_rn(acc, p.scale);
        if constexpr (MODE == kAllReduce) {
#pragma unroll
            for (int r = 0; r < W; ++r) st1(p.a[r] + i, acc);
        } else {
            st1(p.out + i, acc);
        }
    }
}

// The dynamic shared memory of a bulk CTA: S stages of W input tiles and one
// result tile, then the full and empty mbarriers of every stage.
template <int W, int MODE>
struct BulkSmem {
    float *in;        // [S][W][T]
    float *res;       // [S][T]
    uint64_t *full;   // [S]
    uint64_t *empty;  // [S]
};

template <int W, int MODE>
__device__ __forceinline__ BulkSmem<W, MODE> bulk_smem_init(unsigned char *smem)
{
    using Sh = BulkShape<W, MODE>;
    BulkSmem<W, MODE> m;
    m.in = (float *)smem;
    m.res = m.in + (size_t)Sh::S * W * Sh::T;
    m.full = (uint64_t *)(m.res + (size_t)Sh::S * Sh::T);
    m.empty = m.full + Sh::S;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Sh::S; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    return m;
}

// The pipeline of one CTA, after its mbarriers are initialized and visible:
// the producer lane streams the CTA's tiles, the consumer warps fold them
// and store the results, and first fold the call's edges.
template <int W, int MODE>
__device__ __forceinline__ void bulk_run(const BulkParams<W> &p, const BulkSmem<W, MODE> &m)
{
    using Sh = BulkShape<W, MODE>;
    constexpr int T = Sh::T, S = Sh::S, NC = 32 * Sh::NCW;
    float *in = m.in, *res = m.res;
    uint64_t *full = m.full, *empty = m.empty;

    if (threadIdx.x < 32) {  // producer warp: one lane issues the loads
        if (threadIdx.x == 0) {
            long long k = 0;
            for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
                const int s = (int)(k % S);
                if (k >= S && !mbar_wait(&empty[s], (uint32_t)(((k / S) - 1) & 1))) break;
                mbar_arrive_expect(&full[s], W * T * 4);
#pragma unroll
                for (int r = 0; r < W; ++r)
                    bulk_load(in + ((size_t)s * W + r) * T, p.a[r] + p.head + t * T, T * 4, &full[s]);
            }
            // before this CTA may exit, every load it issued has landed
            for (long long j = (k > S ? k - S : 0); j < k; ++j)
                if (!mbar_wait(&full[j % S], (uint32_t)((j / S) & 1))) break;
        }
        return;
    }

    const int tc = threadIdx.x - 32;
    bulk_edges<W, MODE>(p, tc);
    long long k = 0;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
        const int s = (int)(k % S);
        // Each consumer waits (bounded) for the stage itself, which also
        // makes the bulk copy's bytes visible to it. The vote then gives all
        // NC consumers one verdict: if any wait ran out, every consumer
        // leaves the loop here, and none is left at the barrier below.
        const bool landed = mbar_wait(&full[s], (uint32_t)((k / S) & 1));
        if (tc == 0 && landed) bulk_wait_read<S - 1>();  // the store of tile k-S has read res[s]
        if (named_sync_any(1, NC, !landed)) break;
        const float *src = in + (size_t)s * W * T;
        float *dst = res + (size_t)s * T;
        for (int j = tc * 4; j < T; j += NC * 4) {
            float4 acc = *(const float4 *)(src + j);
#pragma unroll
            for (int r = 1; r < W; ++r) {
                const float4 x = *(const float4 *)(src + (size_t)r * T + j);
                acc.x = __fadd_rn(acc.x, x.x);
                acc.y = __fadd_rn(acc.y, x.y);
                acc.z = __fadd_rn(acc.z, x.z);
                acc.w = __fadd_rn(acc.w, x.w);
            }
            if (p.do_scale) {
                acc.x = __fmul_rn(acc.x, p.scale);
                acc.y = __fmul_rn(acc.y, p.scale);
                acc.z = __fmul_rn(acc.z, p.scale);
                acc.w = __fmul_rn(acc.w, p.scale);
            }
            *(float4 *)(dst + j) = acc;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> bulk store
        named_sync(1, NC);
        if (tc == 0) {
            mbar_arrive(&empty[s]);  // the input stage may be refilled
            const int64_t e = p.head + t * T;
            if constexpr (MODE == kAllReduce) {
#pragma unroll
                for (int r = 0; r < W; ++r) bulk_store(p.a[r] + e, dst, T * 4);
            } else {
                bulk_store(p.out + e, dst, T * 4);
            }
            bulk_commit();
        }
    }
    if (tc == 0) bulk_wait_all();
}

template <int W, int MODE>
__global__ void __launch_bounds__(BulkShape<W, MODE>::THREADS) fold_bulk_kernel(const __grid_constant__ BulkParams<W> p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const BulkSmem<W, MODE> m = bulk_smem_init<W, MODE>(smem);
    pdl_enter(p.pdl);
    __syncthreads();
    bulk_run<W, MODE>(p, m);
}

// Elements per thread per iteration of the table kernel's scalar path
// (entries at different 16-byte phases). Measured on GB300 at 2^24 against
// one element per iteration: W=2 and W=4 folds and all-reduces 1.6-3.7x
// faster with 8; the W=8 fold 1.6x faster with 2, while the W=8 all-reduce
// lost 13% with 2 and keeps 1.
#ifndef DETFOLD_TABLE_SCALAR_U
#define DETFOLD_TABLE_SCALAR_U(W, MODE) ((W) <= 4 ? 8 : ((MODE) == kAllReduce ? 1 : 2))
#endif

// A large fold or all-reduce over a device-resident pointer table.
struct BulkTableParams {
    const float *const *table;  // device array of W device pointers
    float *out;                 // sum mode only
    int *status;                // optional device status word
    int64_t len;
    float scale;
    int do_scale;
    int pdl;
};

// The table is read on the device after the wait (the preceding work may
// have written it). Every entry is checked as the other table kernels check
// it (NULL, 4-byte alignment, in rank order, with the status word written
// and nothing else touched on a bad entry). When every entry (and the
// output) shares one 16-byte phase, the CTA runs the same bulk pipeline as
// fold_bulk_kernel; otherwise the grid folds with coalesced scalar accesses.
template <int W, int MODE>
__global__ void __launch_bounds__(BulkShape<W, MODE>::THREADS) fold_bulk_table_kernel(const __grid_constant__ BulkTableParams tp)
{
    constexpr int T = BulkShape<W, MODE>::T;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ BulkParams<W> sp;
    __shared__ int s_code, s_bulk;
    const BulkSmem<W, MODE> m = bulk_smem_init<W, MODE>(smem);
    pdl_enter(tp.pdl);
    if (threadIdx.x == 0) {
        int code = DETFOLD_OK;
        for (int r = 0; r < W; ++r) {
            float *q = const_cast<float *>(tp.table[r]);
            if (code == DETFOLD_OK && q == nullptr) code = DETFOLD_ERR_NULL;
            if (code == DETFOLD_OK && ((uintptr_t)q & 3u)) code = DETFOLD_ERR_ALIGN;
            sp.a[r] = q;
        }
        int bulk = 0;
        if (code == DETFOLD_OK) {
            const uintptr_t ph = (uintptr_t)sp.a[0] & 15u;
            bool same = (MODE == kAllReduce) || ((uintptr_t)tp.out & 15u) == ph;
            for (int r = 1; r < W; ++r) same = same && ((uintptr_t)sp.a[r] & 15u) == ph;
            int64_t head = (int64_t)(((16u - ph) & 15u) / 4u);
            if (head > tp.len) head = tp.len;
            sp.out = tp.out;
            sp.len = tp.len;
            sp.head = head;
            sp.ntiles = (tp.len - head) / T;
            sp.scale = tp.scale;
            sp.do_scale = tp.do_scale;
            sp.pdl = tp.pdl;
            bulk = same && sp.ntiles >= 1;
        }
        s_code = code;
        s_bulk = bulk;
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0 && tp.status) *tp.status = s_code;
    if (s_code != DETFOLD_OK) return;
    if (s_bulk) {
        bulk_run<W, MODE>(sp, m);
        return;
    }
    // entries at different 16-byte phases: coalesced scalar accesses, U
    // elements per thread per iteration with all their loads issued before
    // the chains (each element is read, then written, by the same thread)
    constexpr int U = DETFOLD_TABLE_SCALAR_U(W, MODE);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (U - 1) * stride < tp.len; i += U * stride) {
        float x[U][W];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < W; ++r) x[u][r] = ld1<false>(sp.a[r] + i + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float acc = x[u][0];
#pragma unroll
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, x[u][r]);
            if (tp.do_scale) acc = __fmul_rn(acc, tp.scale);
            if constexpr (MODE == kAllReduce) {
#pragma unroll
                for (int r = 0; r < W; ++r) st1(sp.a[r] + i + u * stride, acc);
            } else {
                st1(tp.out + i + u * stride, acc);
            }
        }
    }
    for (; i < tp.len; i += stride) {
        float acc = ld1<false>(sp.a[0] + i);
#pragma unroll
        for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, ld1<false>(sp.a[r] + i));
        if (tp.do_scale) acc = __fmul_rn(acc, tp.scale);
        if constexpr (MODE == kAllReduce) {
#pragma unroll
            for (int r = 0; r < W; ++r) st1(sp.a[r] + i, acc);
        } else {
            st1(tp.out + i, acc);
        }
    }
}

// ---------------------------------------------------------------- arenas at different 16-byte phases

// The all-reduce when the arenas do not share a 16-byte phase. Tiles follow
// arena 0's 16-byte grid, starting `base` (4..7) elements in. Arena r's
// elements of a tile begin p_r (0..3) elements past a 16-byte boundary, so
// its tile is loaded from that boundary, T + 4 floats long (a whole number
// of 16-byte units), and read at offset p_r in shared memory. The folded
// tile is written to shared memory once unshifted and once per shift
// q = (4 - p_r) mod 4 that some arena needs; arena r's 16-byte-aligned
// interior (T - 4 floats when p_r != 0) then leaves with one bulk store from
// the copy shifted by q_r, and its two partial 16-byte units (q_r and p_r
// elements) with scalar stores. Every element is written once, by the CTA
// that folded it; the elements a tile's loads cover beyond its own range
// are never used, so the update in place needs no ordering between CTAs.
// The call's head [0, base) and tail after the last whole tile are scalar.
template <int W>
struct MixedParams {
    float *a[W];   // the arenas, read and written
    int p[W];      // element phase (0..3) of each arena's tile starts
    int qmask;     // bit q: some arena stores from the copy shifted by q
    int64_t len, base, ntiles;
    float scale;
    int do_scale;
    int pdl;
};

// Shapes from a GB300 sweep (2^24 per arena, identical bits): up to W = 5,
// 4 KB tiles in 2 stages at up to 4 CTAs per SM (as many as shared memory
// holds: 3 from W = 3 on); above, 8 KB tiles in 2 stages at one CTA per SM.
// The limit is the bytes each SM keeps in flight (2 CTAs of 4 KB tiles at
// W = 3 ran 18% slower). DETFOLD_MIXED_T/_S/_C, when defined, override
// every W.
#ifdef DETFOLD_MIXED_T
#define DETFOLD_MIXED_T_OF(W) DETFOLD_MIXED_T
#else
#define DETFOLD_MIXED_T_OF(W) ((W) <= 5 ? 1024 : 2048)
#endif
#ifdef DETFOLD_MIXED_S
#define DETFOLD_MIXED_S_OF(W) DETFOLD_MIXED_S
#else
#define DETFOLD_MIXED_S_OF(W) 2
#endif
#ifdef DETFOLD_MIXED_C
#define DETFOLD_MIXED_C_OF(W) DETFOLD_MIXED_C
#else
#define DETFOLD_MIXED_C_OF(W) ((W) <= 5 ? 4 : 1)
#endif
template <int W>
struct MixedShape {
    static constexpr int T = DETFOLD_MIXED_T_OF(W), S = DETFOLD_MIXED_S_OF(W), CTAS_PER_SM = DETFOLD_MIXED_C_OF(W);
    static constexpr int TL = T + 4;  // floats loaded per arena and tile
    static constexpr int NCW = DETFOLD_BULK_NCW;
    static constexpr int THREADS = 32 * (1 + NCW);
    static constexpr size_t SMEM = (size_t)S * W * TL * 4 + (size_t)S * 4 * T * 4 + 2 * S * 8;
    static_assert(T % 4 == 0 && T >= 8, "tiles of whole 16-byte units, with an interior");
    static_assert(W > 6 || T % (4 * 32 * NCW) == 0, "the consumers cover a tile in whole passes of 4 elements per thread");
    static_assert(8 * W <= 32 * NCW, "one consumer thread per partial element");
};

template <int W>
__global__ void __launch_bounds__(MixedShape<W>::THREADS) fold_bulk_mixed_kernel(const __grid_constant__ MixedParams<W> p)
{
    using Sh = MixedShape<W>;
    constexpr int T = Sh::T, S = Sh::S, TL = Sh::TL, NC = 32 * Sh::NCW;
    extern __shared__ __align__(128) unsigned char smem[];
    float *in = (float *)smem;                          // [S][W][TL]
    float *res = in + (size_t)S * W * TL;               // [S][4][T]: copy q is shifted by q
    uint64_t *full = (uint64_t *)(res + (size_t)S * 4 * T);
    uint64_t *empty = full + S;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_enter(p.pdl);
    __syncthreads();

    if (threadIdx.x < 32) {  // producer warp: one lane issues the loads
        if (threadIdx.x == 0) {
            long long k = 0;
            for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
                const int s = (int)(k % S);
                if (k >= S && !mbar_wait(&empty[s], (uint32_t)(((k / S) - 1) & 1))) break;
                mbar_arrive_expect(&full[s], W * TL * 4);
#pragma unroll
                for (int r = 0; r < W; ++r)
                    bulk_load(in + ((size_t)s * W + r) * TL, p.a[r] + p.base + t * T - p.p[r], TL * 4, &full[s]);
            }
            for (long long j = (k > S ? k - S : 0); j < k; ++j)  // own copies landed
                if (!mbar_wait(&full[j % S], (uint32_t)((j / S) & 1))) break;
        }
        return;
    }

    const int tc = threadIdx.x - 32;
    {   // the call's head and tail, scalar, while the first loads are in flight
        const int64_t tail0 = p.base + p.ntiles * T;
        const int64_t nhead = p.ntiles ? p.base : p.len, ntail = p.ntiles ? p.len - tail0 : 0;
        for (int64_t idx = (int64_t)blockIdx.x * NC + tc; idx < nhead + ntail; idx += (int64_t)gridDim.x * NC) {
            const int64_t e = idx < nhead ? idx : tail0 + (idx - nhead);
            float acc = ld1<false>(p.a[0] + e);
#pragma unroll
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, ld1<false>(p.a[r] + e));
            if (p.do_scale) acc = __fmul_rn(acc, p.scale);
#pragma unroll
            for (int r = 0; r < W; ++r) st1(p.a[r] + e, acc);
        }
    }
    long long k = 0;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
        const int s = (int)(k % S);
        // each consumer waits (bounded) for the stage; the vote gives all
        // consumers one verdict (as in bulk_run)
        const bool landed = mbar_wait(&full[s], (uint32_t)((k / S) & 1));
        if (tc == 0 && landed) bulk_wait_read<S - 1>();  // the stores of tile k-S have read res[s]
        if (named_sync_any(1, NC, !landed)) break;
        const float *src = in + (size_t)s * W * TL;
        float *rq = res + (size_t)s * 4 * T;
        if constexpr (W <= 6) {
            // thread tc takes elements e0 + tc + m * NC: a warp's shared loads
            // and stores are 32 consecutive words, free of bank conflicts
            // whatever the arena's phase offset (measured 0.4-3.9% faster
            // for W = 2..6 at 2^24 per arena)
            for (int e0 = 0; e0 < T; e0 += NC * 4) {
                float acc[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) acc[m] = src[p.p[0] + e0 + m * NC + tc];
#pragma unroll
                for (int r = 1; r < W; ++r)
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        acc[m] = __fadd_rn(acc[m], src[(size_t)r * TL + p.p[r] + e0 + m * NC + tc]);
                if (p.do_scale) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc[m] = __fmul_rn(acc[m], p.scale);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) rq[e0 + m * NC + tc] = acc[m];
#pragma unroll
                for (int q = 1; q < 4; ++q) {
                    if (p.qmask & (1 << q)) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int e = e0 + m * NC + tc;  // copy q holds elements q .. T-5+q
                            if (e >= q && e < T - 4 + q) rq[q * T + e - q] = acc[m];
                        }
                    }
                }
            }
        } else {
            // W = 7, 8: four consecutive elements per thread and one 16-byte
            // store of copy 0 (measured 1.3-2.2% faster here than the layout
            // above, despite its 4-way bank conflicts)
            for (int j = tc * 4; j < T; j += NC * 4) {
                float acc[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) acc[kk] = src[p.p[0] + j + kk];
#pragma unroll
                for (int r = 1; r < W; ++r)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) acc[kk] = __fadd_rn(acc[kk], src[(size_t)r * TL + p.p[r] + j + kk]);
                if (p.do_scale) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) acc[kk] = __fmul_rn(acc[kk], p.scale);
                }
                *(float4 *)(rq + j) = make_float4(acc[0], acc[1], acc[2], acc[3]);
#pragma unroll
                for (int q = 1; q < 4; ++q) {
                    if (p.qmask & (1 << q)) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int e = j + kk;  // copy q holds elements q .. T-5+q
                            if (e >= q && e < T - 4 + q) rq[q * T + e - q] = acc[kk];
                        }
                    }
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> bulk store
        named_sync(1, NC);
        const int64_t ts = p.base + t * T;
        if (tc < 8 * W) {  // the partial 16-byte units at the tile's two ends
            const int r = tc >> 3, kk = tc & 7, pr = p.p[r], qr = (4 - pr) & 3;
            const int e = kk < 4 ? (kk < qr ? kk : -1) : (kk - 4 < pr ? T - pr + (kk - 4) : -1);
            if (e >= 0) st1(p.a[r] + ts + e, rq[e]);
        }
        if (tc == 0) {
            mbar_arrive(&empty[s]);  // the input stage may be refilled
#pragma unroll
            for (int r = 0; r < W; ++r) {
                const int qr = (4 - p.p[r]) & 3;
                bulk_store(p.a[r] + ts + qr, rq + (size_t)qr * T, (qr ? T - 4 : T) * 4);
            }
            bulk_commit();
        }
    }
    if (tc == 0) bulk_wait_all();
}

// Shared-memory opt-in, resident CTAs and the per-CTA shared-memory request
// (exclusive_smem), once per kernel and device.
template <auto Kernel, typename Sh>
cudaError_t bulk_grid_of(int *grid, int *smem_bytes)
{
    static std::atomic<int> cache[64], cache_smem[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int v = cache[dev].load(std::memory_order_acquire);
    if (v <= 0) {
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, Kernel, Sh::THREADS, Sh::SMEM);
        if (e != cudaSuccess) return e;
        if (Sh::CTAS_PER_SM > 0 && per_sm > Sh::CTAS_PER_SM) per_sm = Sh::CTAS_PER_SM;
        if (per_sm < 1) per_sm = 1;
        size_t smem = Sh::SMEM;
        e = exclusive_smem(dev, Sh::SMEM, per_sm, &smem);
        if (e != cudaSuccess) return e;
        if (smem != Sh::SMEM) {
            e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        cache_smem[dev].store((int)smem, std::memory_order_relaxed);
        v = sms * per_sm;
        cache[dev].store(v, std::memory_order_release);
    }
    *grid = v;
    *smem_bytes = cache_smem[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
}

template <int W, int MODE>
cudaError_t launch_bulk_fixed(const LaunchSpec &s, int64_t head, cudaStream_t stream)
{
    using Sh = BulkShape<W, MODE>;
    BulkParams<W> p = {};
    for (int r = 0; r < W; ++r) p.a[r] = const_cast<float *>(s.src[r]);
    p.out = s.out;
    p.len = s.len;
    p.head = head;
    p.ntiles = (s.len - head) / Sh::T;
    p.scale = s.scale;
    p.do_scale = s.do_scale;
    p.pdl = DETFOLD_PDL_ALL ? 1 : 0;
    int cap = 0, smem = 0;
    cudaError_t e = bulk_grid_of<fold_bulk_kernel<W, MODE>, BulkShape<W, MODE>>(&cap, &smem);
    if (e != cudaSuccess) return e;
    int64_t grid = p.ntiles < cap ? p.ntiles : cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(Sh::THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fold_bulk_kernel<W, MODE>, p);
}

template <int W, int MODE>
cudaError_t launch_bulk_table_fixed(const BulkTableParams &tp, cudaStream_t stream)
{
    using Sh = BulkShape<W, MODE>;
    int cap = 0, smem = 0;
    cudaError_t e = bulk_grid_of<fold_bulk_table_kernel<W, MODE>, BulkShape<W, MODE>>(&cap, &smem);
    if (e != cudaSuccess) return e;
    int64_t grid = tp.len / Sh::T;  // about one CTA per tile, at most the resident CTAs
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(Sh::THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (tp.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fold_bulk_table_kernel<W, MODE>, tp);
}

template <int W>
cudaError_t launch_bulk_mixed_fixed(const LaunchSpec &s, cudaStream_t stream)
{
    using Sh = MixedShape<W>;
    MixedParams<W> p = {};
    const int64_t head0 = (4 - elem_phase(s.src[0], 4)) % 4;
    p.base = head0 + 4;
    p.len = s.len;
    p.ntiles = s.len >= p.base + 4 + Sh::T ? (s.len - p.base - 4) / Sh::T : 0;
    for (int r = 0; r < W; ++r) {
        p.a[r] = const_cast<float *>(s.src[r]);
        p.p[r] = elem_phase(s.src[r] + p.base, 4);
        p.qmask |= 1 << ((4 - p.p[r]) & 3);
    }
    p.scale = s.scale;
    p.do_scale = s.do_scale;
    p.pdl = DETFOLD_PDL_ALL ? 1 : 0;
    int cap = 0, smem = 0;
    cudaError_t e = bulk_grid_of<fold_bulk_mixed_kernel<W>, Sh>(&cap, &smem);
    if (e != cudaSuccess) return e;
    int64_t grid = p.ntiles < cap ? p.ntiles : cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(Sh::THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fold_bulk_mixed_kernel<W>, p);
}

template <int MODE>
cudaError_t launch_bulk_table_mode(const BulkTableParams &tp, int W, cudaStream_t stream)
{
    switch (W) {
    case 1: return launch_bulk_table_fixed<1, MODE>(tp, stream);
    case 2: return launch_bulk_table_fixed<2, MODE>(tp, stream);
    case 3: return launch_bulk_table_fixed<3, MODE>(tp, stream);
    case 4: return launch_bulk_table_fixed<4, MODE>(tp, stream);
    case 5: return launch_bulk_table_fixed<5, MODE>(tp, stream);
    case 6: return launch_bulk_table_fixed<6, MODE>(tp, stream);
    case 7: return launch_bulk_table_fixed<7, MODE>(tp, stream);
    default: return launch_bulk_table_fixed<8, MODE>(tp, stream);
    }
}

template <int MODE>
cudaError_t launch_bulk_mode(const LaunchSpec &s, int64_t head, cudaStream_t stream)
{
    switch (s.W) {
    case 1: return launch_bulk_fixed<1, MODE>(s, head, stream);
    case 2: return launch_bulk_fixed<2, MODE>(s, head, stream);
    case 3: return launch_bulk_fixed<3, MODE>(s, head, stream);
    case 4: return launch_bulk_fixed<4, MODE>(s, head, stream);
    case 5: return launch_bulk_fixed<5, MODE>(s, head, stream);
    case 6: return launch_bulk_fixed<6, MODE>(s, head, stream);
    case 7: return launch_bulk_fixed<7, MODE>(s, head, stream);
    default: return launch_bulk_fixed<8, MODE>(s, head, stream);
    }
}

}  // namespace

cudaError_t read_pipeline_timeouts_bulk(unsigned long long *count) { return read_unit_timeouts(count); }

template <int MODE>
int tile_floats_of(int W)
{
    switch (W) {
    case 1: return BulkShape<1, MODE>::T;
    case 2: return BulkShape<2, MODE>::T;
    case 3: return BulkShape<3, MODE>::T;
    case 4: return BulkShape<4, MODE>::T;
    case 5: return BulkShape<5, MODE>::T;
    case 6: return BulkShape<6, MODE>::T;
    case 7: return BulkShape<7, MODE>::T;
    default: return BulkShape<8, MODE>::T;
    }
}

int bulk_tile_floats(int W, int mode)
{
    return mode == kAllReduce ? tile_floats_of<kAllReduce>(W) : tile_floats_of<kSumCoherent>(W);
}

cudaError_t launch_bulk_table(const float *const *d_table, float *out, int *d_status, int W, int64_t len,
                              float scale, int do_scale, int mode, cudaStream_t stream)
{
    BulkTableParams tp = {};
    tp.table = d_table;
    tp.out = out;
    tp.status = d_status;
    tp.len = len;
    tp.scale = scale;
    tp.do_scale = do_scale;
    tp.pdl = DETFOLD_PDL_ALL ? 1 : 0;
    if (mode == kAllReduce) return launch_bulk_table_mode<kAllReduce>(tp, W, stream);
    return launch_bulk_table_mode<kSumCoherent>(tp, W, stream);
}

cudaError_t launch_bulk_mixed(const LaunchSpec &s, cudaStream_t stream)
{
    switch (s.W) {
    case 1: return launch_bulk_mixed_fixed<1>(s, stream);
    case 2: return launch_bulk_mixed_fixed<2>(s, stream);
    case 3: return launch_bulk_mixed_fixed<3>(s, stream);
    case 4: return launch_bulk_mixed_fixed<4>(s, stream);
    case 5: return launch_bulk_mixed_fixed<5>(s, stream);
    case 6: return launch_bulk_mixed_fixed<6>(s, stream);
    case 7: return launch_bulk_mixed_fixed<7>(s, stream);
    default: return launch_bulk_mixed_fixed<8>(s, stream);
    }
}

cudaError_t launch_bulk(const LaunchSpec &s, int64_t head, cudaStream_t stream)
{
    if (s.mode == kAllReduce) return launch_bulk_mode<kAllReduce>(s, head, stream);
    return launch_bulk_mode<kSumCoherent>(s, head, stream);
}


}  // namespace detfold
