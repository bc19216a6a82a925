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
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold_launch.cuh"

namespace detfold {

namespace {

template <int VEC>
__global__ void __launch_bounds__(256) move_pairs_kernel(const __grid_constant__ MoveParams p)
{
    constexpr int G = 4;
    pdl_enter(p.pdl);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
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
    // head and tail elements (fewer than VEC each)
    const int64_t tail0 = p.head + p.nvec * VEC;
    const int64_t ntail = p.len - tail0;
    for (int part = 0; part < 2; ++part) {
        const int64_t i = part == 0 ? gtid : tail0 + gtid;
        if ((part == 0 && gtid < p.head) || (part == 1 && gtid < ntail)) {
            for (int k = 0; k < p.K; ++k) st1(p.dst[k] + i, ld1<true>(p.src[k] + i));
        }
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
    MoveParams p = {};
    for (int k = 0; k < K; ++k) {
        p.src[k] = src[k];
        p.dst[k] = dst[k];
    }
    p.K = K;
    p.len = len;
    const bool small = len <= DETFOLD_SMALL_LEN;
    p.pdl = (small && DETFOLD_SMALL_PDL) ? 1 : 0;
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
    if (vec == 8) return launch_kernel<move_pairs_kernel<8>>(p, p.nvec, 1, small, 256, 0, stream);
    if (vec == 4) return launch_kernel<move_pairs_kernel<4>>(p, p.nvec, 1, small, 256, 0, stream);
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

}  // namespace detfold
