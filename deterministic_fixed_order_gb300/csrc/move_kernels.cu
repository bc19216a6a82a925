// Pure byte movement on one device: K (source -> destination) pairs of equal
// length in one launch. No arithmetic touches the values, so every
// destination receives the source's bits exactly (memra-engine 0.128.0
// tests/tp_ar_gpu.rs, `broadcast_and_all_gather_move_bytes_exactly`: the
// hops of the TP walk move bytes and nothing else).
//
// Uses: the staged comparator's exchange (every rank's shard slice into its
// stack slot) and distribute (the owner's shard to every other arena --
// consecutive pairs with the same source read it once), and the public
// broadcast and all-gather.
//
// Each thread loads the vectors of up to G pairs before storing any of them.
// Sources are read through the read-only path: the API layer guarantees that
// no destination overlaps any source of the same launch.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold_async.cuh"
#include "detfold_launch.cuh"

namespace detfold {

namespace {

// ---------------------------------------------------------------- bulk-async movement

// Large aligned moves: one loader lane streams a tile of every distinct
// source (consecutive pairs with the same source share it) into a ring of
// shared-memory stages with cp.async.bulk; one storer lane issues a bulk
// store per destination straight from shared memory, so a source with
// several destinations (a distribute phase, a broadcast) is read from DRAM
// once. A stage is released only after the stores reading it have finished
// reading (wait_group.read). Waits are bounded (detfold_async.cuh).
#ifndef DETFOLD_MOVE_T
#define DETFOLD_MOVE_T 2048  // floats per source per tile (8 KB)
#endif
#ifndef DETFOLD_MOVE_S_LO
#define DETFOLD_MOVE_S_LO 4  // stages, up to 4 distinct sources
#endif
#ifndef DETFOLD_MOVE_S_HI
#define DETFOLD_MOVE_S_HI 2  // stages, more sources
#endif
#ifndef DETFOLD_MOVE_CTAS_PER_SM
#define DETFOLD_MOVE_CTAS_PER_SM 4
#endif
#ifndef DETFOLD_MOVE_CTAS_PER_SM_G1
#define DETFOLD_MOVE_CTAS_PER_SM_G1 2  // single-source launches (broadcast, the staged distribute)
#endif
template <int G>
struct MoveShape {
    static constexpr int T = DETFOLD_MOVE_T;
    static constexpr int S = G <= 4 ? DETFOLD_MOVE_S_LO : DETFOLD_MOVE_S_HI;
    static constexpr size_t SMEM = (size_t)S * G * T * 4 + 2 * S * 8;
    static_assert(T % 4 == 0, "tiles are whole 16-byte vectors");
};

template <int G>
struct MoveBulkParams {
    const float *src[G];           // distinct sources
    float *dst[kMaxPairs];         // destinations in pair order
    unsigned char grp[kMaxPairs];  // pair -> source slot
    int K;
    int pdl;
    int64_t len, head, ntiles;
};

template <int G>
__global__ void __launch_bounds__(64) move_bulk_kernel(const __grid_constant__ MoveBulkParams<G> p)
{
    using Sh = MoveShape<G>;
    constexpr int T = Sh::T, S = Sh::S;
    extern __shared__ __align__(128) unsigned char smem[];
    float *buf = (float *)smem;  // [S][G][T]
    uint64_t *full = (uint64_t *)(buf + (size_t)S * G * T);
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
    if (threadIdx.x == 0) {  // loader
        long long k = 0;
        for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
            const int s = (int)(k % S);
            if (k >= S && !mbar_wait(&empty[s], (uint32_t)(((k / S) - 1) & 1))) break;
            mbar_arrive_expect(&full[s], G * T * 4);
#pragma unroll
            for (int g = 0; g < G; ++g)
                bulk_load(buf + ((size_t)s * G + g) * T, p.src[g] + p.head + t * T, T * 4, &full[s]);
        }
        for (long long j = (k > S ? k - S : 0); j < k; ++j)  // own copies landed
            if (!mbar_wait(&full[j % S], (uint32_t)((j / S) & 1))) break;
        return;
    }
    if (threadIdx.x == 32) {  // storer
        long long k = 0;
        for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++k) {
            const int s = (int)(k % S);
            if (!mbar_wait(&full[s], (uint32_t)((k / S) & 1))) break;
            const int64_t e = p.head + t * T;
            for (int q = 0; q < p.K; ++q) bulk_store(p.dst[q] + e, buf + ((size_t)s * G + p.grp[q]) * T, T * 4);
            bulk_commit();
            if (k >= 1) {
                bulk_wait_read<1>();              // stores of tile k-1 have read their stage
                mbar_arrive(&empty[(k - 1) % S]);
            }
        }
        bulk_wait_all();
    } else {
        // The 62 other threads move what lies outside the whole tiles: the
        // tail [head + ntiles*T, len) starts 16-byte aligned and goes in
        // 16-byte vectors, one per thread, from the last CTA (the CTAs at the
        // end hold the fewest tiles); the head [0, head) and the tail's last
        // few elements (fewer than 4 each) are scalar, in the last CTA.
        constexpr int NE = 62;
        const int et = threadIdx.x < 32 ? threadIdx.x - 1 : threadIdx.x - 2;
        const int64_t tail0 = p.head + p.ntiles * T;
        const int64_t nv = (p.len - tail0) / 4;
        for (int64_t v = (int64_t)(gridDim.x - 1 - blockIdx.x) * NE + et; v < nv; v += (int64_t)gridDim.x * NE) {
            const int64_t e = tail0 + v * 4;
            for (int k = 0; k < p.K; ++k) stv<4>(p.dst[k] + e, ldv<4, true>(p.src[p.grp[k]] + e));
        }
        if (blockIdx.x == gridDim.x - 1) {
            const int64_t rest0 = tail0 + nv * 4;
            const int nhead = (int)p.head, nrest = (int)(p.len - rest0);
            if (et < nhead + nrest) {
                const int64_t i = et < nhead ? et : rest0 + (et - nhead);
                for (int k = 0; k < p.K; ++k) st1(p.dst[k] + i, ld1<true>(p.src[p.grp[k]] + i));
            }
        }
    }
}

template <int G>
cudaError_t launch_move_bulk_fixed(const float *const *src, float *const *dst, int K, int64_t len,
                                   int64_t head, cudaStream_t stream)
{
    using Sh = MoveShape<G>;
    MoveBulkParams<G> p = {};
    int g = -1;
    for (int k = 0; k < K; ++k) {
        if (k == 0 || src[k] != src[k - 1]) p.src[++g] = src[k];
        p.dst[k] = dst[k];
        p.grp[k] = (unsigned char)g;
    }
    p.K = K;
    p.pdl = DETFOLD_PDL_ALL ? 1 : 0;
    p.len = len;
    p.head = head;
    p.ntiles = (len - head) / Sh::T;
    // resident CTAs (at most DETFOLD_MOVE_CTAS_PER_SM) and the per-CTA shared-memory request
    // that keeps every SM at that count (exclusive_smem), once per device
    static std::atomic<int> cache[64], cache_smem[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int cap = cache[dev].load(std::memory_order_acquire);
    if (cap <= 0) {
        e = cudaFuncSetAttribute(move_bulk_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, move_bulk_kernel<G>, 64, Sh::SMEM);
        if (e != cudaSuccess) return e;
        // one source: 2 CTAs per SM measured 6272 -> 6624 GB/s for a 1:1
        // broadcast and 5942 -> 6059 for 1:3 (2^26), 1:7 unchanged
        const int cap_sm = G == 1 ? DETFOLD_MOVE_CTAS_PER_SM_G1 : DETFOLD_MOVE_CTAS_PER_SM;
        if (per_sm > cap_sm) per_sm = cap_sm;
        if (per_sm < 1) per_sm = 1;
        size_t smem = Sh::SMEM;
        e = exclusive_smem(dev, Sh::SMEM, per_sm, &smem);
        if (e != cudaSuccess) return e;
        if (smem != Sh::SMEM) {
            e = cudaFuncSetAttribute(move_bulk_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        cache_smem[dev].store((int)smem, std::memory_order_relaxed);
        cap = sms * per_sm;
        cache[dev].store(cap, std::memory_order_release);
    }
    int64_t grid = p.ntiles < cap ? p.ntiles : cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(64, 1, 1);
    cfg.dynamicSmemBytes = (size_t)cache_smem[dev].load(std::memory_order_relaxed);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, move_bulk_kernel<G>, p);
}

// The head and tail elements of every pair (fewer than VEC each), run by
// the launch's leading p.edge_blocks CTAs, so their memory round trips run
// beside the vectors' instead of after them. Element j of the K * nedge
// numbers pair j / nedge; thread `i` takes j = i, i + step, ..., four loads
// ahead of their stores.
template <int VEC>
__device__ __forceinline__ void move_edges(const MoveParams &p, int i, int step)
{
    const int nedge = (int)(p.len - p.nvec * VEC);  // head + tail
    const int64_t tail0 = p.head + p.nvec * VEC;
    const int n = p.K * nedge;
    for (; i < n; i += 4 * step) {
        float x[4];
        int64_t e[4];
        int k[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = i + u * step;
            k[u] = j < n ? j / nedge : 0;
            const int q = j - k[u] * nedge;
            e[u] = q < (int)p.head ? q : tail0 + (q - (int)p.head);
            if (j < n) x[u] = ld1<true>(p.src[k[u]] + e[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i + u * step < n) st1(p.dst[k[u]] + e[u], x[u]);
    }
}

template <int VEC>
__global__ void __launch_bounds__(256) move_pairs_kernel(const __grid_constant__ MoveParams p)
{
    constexpr int G = 4;
    pdl_enter(p.pdl);
    if ((int)blockIdx.x < p.edge_blocks) {
        move_edges<VEC>(p, blockIdx.x * blockDim.x + threadIdx.x, p.edge_blocks * blockDim.x);
        return;
    }
    const int64_t stride = (int64_t)(gridDim.x - p.edge_blocks) * blockDim.x;
    const int64_t gtid = (int64_t)(blockIdx.x - p.edge_blocks) * blockDim.x + threadIdx.x;
    for (int64_t v = gtid; v < p.nvec; v += stride) {
        const int64_t e = p.head + v * VEC;
        Vec<VEC> x[G];
        for (int k0 = 0; k0 < p.K; k0 += G) {
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const int kk = k0 + k;
                if (kk < p.K) {
                    if (kk > 0 && p.src[kk] == p.src[kk - 1])
                        x[k] = x[(k + G - 1) % G];  // same source as the previous pair
                    else
                        x[k] = ldv<VEC, true>(p.src[kk] + e);
                }
            }
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (k0 + k < p.K) stv<VEC>(p.dst[k0 + k] + e, x[k]);
        }
    }
}

// Small moves (len <= DETFOLD_SMALL_LEN, every pointer at one phase): one
// (pair, vector) per thread with 32-bit indices, so a call is one dependent
// load and store, not one per group of pairs as in the looping kernel above.
// Pairs that share a source load it separately (from L2, at these sizes).
// EDGES: the call has a head or a tail, moved by the leading p.edge_blocks
// CTAs (one element per thread); without, the kernel has no edge code.
template <int VEC, bool EDGES>
__global__ void __launch_bounds__(DETFOLD_SMALL_THREADS) move_small_kernel(const __grid_constant__ MoveParams p)
{
    static_assert((int64_t)DETFOLD_SMALL_LEN * kMaxPairs < (1LL << 31), "small-move indices are 32-bit");
    pdl_enter(p.pdl);
    int b = blockIdx.x;
    if constexpr (EDGES) {
        if (b < p.edge_blocks) {
            move_edges<VEC>(p, b * blockDim.x + threadIdx.x, p.edge_blocks * blockDim.x);
            return;
        }
        b -= p.edge_blocks;
    }
    const int i = b * blockDim.x + threadIdx.x;
    const int nvec = (int)p.nvec;
    if (i < p.K * nvec) {
        const int k = i / nvec;
        const int e = (int)p.head + (i - k * nvec) * VEC;
        stv<VEC>(p.dst[k] + e, ldv<VEC, true>(p.src[k] + e));
    }
}

// Operands at different 4-byte phases: coalesced scalar moves.
__global__ void __launch_bounds__(256) move_pairs_scalar_kernel(const __grid_constant__ MoveParams p)
{
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.len; i += stride) {
        float x = 0.0f;
        for (int k = 0; k < p.K; ++k) {
            if (k == 0 || p.src[k] != p.src[k - 1]) x = ld1<true>(p.src[k] + i);
            st1(p.dst[k] + i, x);
        }
    }
}

int elem_phase_any(const void *q, int vec) { return (int)(((uintptr_t)q % (uintptr_t)(vec * 4)) / 4); }

}  // namespace

static cudaError_t launch_move_chunk(const float *const *src, float *const *dst, int K,
                                     int64_t len, cudaStream_t stream)
{
    // bulk-async path: large, every operand at one 16-byte phase, <= 8 distinct sources
    if (DETFOLD_USE_BULK && DETFOLD_USE_BULK_MOVE && len >= DETFOLD_BULK_MOVE_MIN_LEN) {
        int groups = 0;
        for (int k = 0; k < K; ++k) groups += (k == 0 || src[k] != src[k - 1]);
        const int ph = elem_phase_any(src[0], 4);
        bool same = true;
        for (int k = 0; same && k < K; ++k)
            same = elem_phase_any(src[k], 4) == ph && elem_phase_any(dst[k], 4) == ph;
        const int64_t head = (4 - ph) % 4;
        if (same && groups <= 8 && len - head >= MoveShape<1>::T) {
            switch (groups) {
            case 1: return launch_move_bulk_fixed<1>(src, dst, K, len, head, stream);
            case 2: return launch_move_bulk_fixed<2>(src, dst, K, len, head, stream);
            case 3: return launch_move_bulk_fixed<3>(src, dst, K, len, head, stream);
            case 4: return launch_move_bulk_fixed<4>(src, dst, K, len, head, stream);
            case 5: return launch_move_bulk_fixed<5>(src, dst, K, len, head, stream);
            case 6: return launch_move_bulk_fixed<6>(src, dst, K, len, head, stream);
            case 7: return launch_move_bulk_fixed<7>(src, dst, K, len, head, stream);
            default: return launch_move_bulk_fixed<8>(src, dst, K, len, head, stream);
            }
        }
    }
    MoveParams p = {};
    for (int k = 0; k < K; ++k) {
        p.src[k] = src[k];
        p.dst[k] = dst[k];
    }
    p.K = K;
    p.len = len;
    const bool small = len <= DETFOLD_SMALL_LEN;
    p.pdl = ((small && DETFOLD_SMALL_PDL) || DETFOLD_PDL_ALL) ? 1 : 0;
    int vec = 0;
    for (int cand : {8, 4}) {
        const int ph = elem_phase_any(src[0], cand);
        bool same = true;
        for (int k = 0; same && k < K; ++k)
            same = elem_phase_any(src[k], cand) == ph && elem_phase_any(dst[k], cand) == ph;
        if (same) {
            vec = cand;
            int64_t head = (cand - ph) % cand;
            if (head > len) head = len;
            p.head = head;
            p.nvec = (len - head) / cand;
            break;
        }
    }
    const int64_t edges = vec ? (int64_t)K * (len - p.nvec * vec) : 0;  // head + tail elements
    if (small && vec != 0) {
        // one thread per (pair, vector), after leading CTAs with one thread
        // per edge element
        p.edge_blocks = (short)((edges + DETFOLD_SMALL_THREADS - 1) / DETFOLD_SMALL_THREADS);  // <= 28
        const int64_t work = (int64_t)K * p.nvec;
        const int eb = p.edge_blocks;
        if (vec == 8)
            return eb ? launch_kernel<move_small_kernel<8, true>>(p, work, 1, true, 256, 0, stream, true, eb)
                      : launch_kernel<move_small_kernel<8, false>>(p, work, 1, true, 256, 0, stream);
        return eb ? launch_kernel<move_small_kernel<4, true>>(p, work, 1, true, 256, 0, stream, true, eb)
                  : launch_kernel<move_small_kernel<4, false>>(p, work, 1, true, 256, 0, stream);
    }
    p.edge_blocks = edges > 0 ? 1 : 0;
    if (vec == 8) return launch_kernel<move_pairs_kernel<8>>(p, p.nvec, 1, small, 256, 0, stream, true, p.edge_blocks);
    if (vec == 4) return launch_kernel<move_pairs_kernel<4>>(p, p.nvec, 1, small, 256, 0, stream, true, p.edge_blocks);
    return launch_kernel<move_pairs_scalar_kernel>(p, len, 1, small, 256, 0, stream);
}

cudaError_t launch_move(const float *const *src, float *const *dst, int K, int64_t len,
                        cudaStream_t stream)
{
    if (K <= 0 || len <= 0) return cudaSuccess;
    for (int k0 = 0; k0 < K; k0 += kMaxPairs) {
        const int n = (K - k0) < kMaxPairs ? (K - k0) : kMaxPairs;
        const cudaError_t e = launch_move_chunk(src + k0, dst + k0, n, len, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_pipeline_timeouts_move(unsigned long long *count) { return read_unit_timeouts(count); }

}  // namespace detfold
