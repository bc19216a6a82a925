// Fold and all-reduce over a pointer table that lives in device memory.
//
// The table is read by the kernel when it runs, so a CUDA graph captured
// once follows new arena addresses written into the table between replays
// (the rebind pattern of memra-engine 0.136.0 tests/gdn_packed_gpu.rs,
// `packed_matches_per_row` with graph_rebind). The arithmetic is the same
// ascending-rank __fadd_rn chain as the other folds (mamba-rs 0.6.2
// src/dist/reducer.rs, `reduce_sum_reference`), so the bits are the same.
//
// The host cannot see the table, so the kernel checks it: every entry must
// be non-NULL and 4-byte aligned, else the kernel writes DETFOLD_ERR_NULL or
// DETFOLD_ERR_ALIGN to the optional status word and touches nothing else.
// The access width (32-byte, 16-byte or scalar) is chosen on the device from
// the entries' phases. Loads are ordinary (coherent) loads: a sum's output
// may be one of the sources.
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold.h"
#include "detfold_launch.cuh"

namespace detfold {

namespace {

struct TableParams {
    const float *const *table;  // device array of W device pointers
    float *out;                 // sum mode only
    int *status;                // optional device status word
    int64_t len;
    float scale;
    int do_scale;
    int W;
    int pdl;
};

__device__ __forceinline__ int phase_of(const void *q, int vec)
{
    return (int)(((uintptr_t)q % (uintptr_t)(vec * 4)) / 4);
}

template <int VEC, int MODE>
__device__ __forceinline__ void table_vec_body(const TableParams &p, const float *const *src,
                                               int64_t head)
{
    constexpr int G = 32 / VEC;
    const int64_t nvec = (p.len - head) / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t v = gtid; v < nvec; v += stride) {
        const int64_t e = head + v * VEC;
        Vec<VEC> acc = ldv<VEC, false>(src[0] + e);
        for (int r0 = 1; r0 < p.W; r0 += G) {
            Vec<VEC> x[G];
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (r0 + k < p.W) x[k] = ldv<VEC, false>(src[r0 + k] + e);
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (r0 + k < p.W)
#pragma unroll
                    for (int j = 0; j < VEC; ++j) acc.v[j] = __fadd_rn(acc.v[j], x[k].v[j]);
        }
        if (p.do_scale) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc.v[j] = __fmul_rn(acc.v[j], p.scale);
        }
        if constexpr (MODE == kAllReduce) {
            for (int r = 0; r < p.W; ++r) stv<VEC>(const_cast<float *>(src[r]) + e, acc);
        } else {
            stv<VEC>(p.out + e, acc);
        }
    }
    // head and tail (fewer than VEC elements each), scalar
    const int64_t tail0 = head + nvec * VEC;
    for (int part = 0; part < 2; ++part) {
        const int64_t i = part == 0 ? gtid : tail0 + gtid;
        if ((part == 0 && gtid < head) || (part == 1 && gtid < p.len - tail0)) {
            float acc = ld1<false>(src[0] + i);
            for (int r = 1; r < p.W; ++r) acc = __fadd_rn(acc, ld1<false>(src[r] + i));
            if (p.do_scale) acc = __fmul_rn(acc, p.scale);
            if constexpr (MODE == kAllReduce) {
                for (int r = 0; r < p.W; ++r) st1(const_cast<float *>(src[r]) + i, acc);
            } else {
                st1(p.out + i, acc);
            }
        }
    }
}

template <int MODE>
__device__ __forceinline__ void table_scalar_body(const TableParams &p, const float *const *src)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.len; i += stride) {
        float acc = ld1<false>(src[0] + i);
        for (int r0 = 1; r0 < p.W; r0 += 8) {
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < p.W) x[k] = ld1<false>(src[r0 + k] + i);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < p.W) acc = __fadd_rn(acc, x[k]);
        }
        if (p.do_scale) acc = __fmul_rn(acc, p.scale);
        if constexpr (MODE == kAllReduce) {
            for (int r = 0; r < p.W; ++r) st1(const_cast<float *>(src[r]) + i, acc);
        } else {
            st1(p.out + i, acc);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(256) fold_table_kernel(const __grid_constant__ TableParams p)
{
    __shared__ const float *s_src[kGenericW];
    __shared__ int s_code, s_vec;
    __shared__ long long s_head;
    // The table may have been written by the preceding work on the stream.
    pdl_enter(p.pdl);
    for (int r = threadIdx.x; r < p.W; r += blockDim.x) s_src[r] = p.table[r];
    __syncthreads();
    if (threadIdx.x == 0) {
        int code = DETFOLD_OK;
        for (int r = 0; r < p.W && code == DETFOLD_OK; ++r) {
            if (s_src[r] == nullptr)
                code = DETFOLD_ERR_NULL;
            else if ((uintptr_t)s_src[r] & 3u)
                code = DETFOLD_ERR_ALIGN;
        }
        int vec = 0;
        long long head = 0;
        if (code == DETFOLD_OK) {
            const int cands[2] = {8, 4};
            for (int c = 0; c < 2 && vec == 0; ++c) {
                const int cand = cands[c];
                const int ph = phase_of(s_src[0], cand);
                bool same = (MODE == kAllReduce) || phase_of(p.out, cand) == ph;
                for (int r = 1; same && r < p.W; ++r) same = phase_of(s_src[r], cand) == ph;
                if (same) {
                    vec = cand;
                    head = (cand - ph) % cand;
                    if (head > p.len) head = p.len;
                }
            }
        }
        s_code = code;
        s_vec = vec;
        s_head = head;
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) *p.status = s_code;
    if (s_code != DETFOLD_OK) return;
    if (s_vec == 8)
        table_vec_body<8, MODE>(p, s_src, s_head);
    else if (s_vec == 4)
        table_vec_body<4, MODE>(p, s_src, s_head);
    else
        table_scalar_body<MODE>(p, s_src);
}

// Small payloads with W <= 8: every thread reads the (broadcast) table
// entries into registers, checks them and picks the access width itself --
// no shared memory and no block barrier between the table load and the data
// loads, which is what the latency of a graph of small folds is made of.
template <int WT, int VEC, int MODE>
__device__ __forceinline__ void table_fixed_vec(const TableParams &p, const float *const (&src)[WT],
                                                int64_t head)
{
    const int64_t nvec = (p.len - head) / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t v = gtid; v < nvec; v += stride) {
        const int64_t e = head + v * VEC;
        Vec<VEC> x[WT];
#pragma unroll
        for (int r = 0; r < WT; ++r) x[r] = ldv<VEC, false>(src[r] + e);
        Vec<VEC> acc = x[0];
#pragma unroll
        for (int r = 1; r < WT; ++r)
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc.v[j] = __fadd_rn(acc.v[j], x[r].v[j]);
        if (p.do_scale) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc.v[j] = __fmul_rn(acc.v[j], p.scale);
        }
        if constexpr (MODE == kAllReduce) {
#pragma unroll
            for (int r = 0; r < WT; ++r) stv<VEC>(const_cast<float *>(src[r]) + e, acc);
        } else {
            stv<VEC>(p.out + e, acc);
        }
    }
    const int64_t tail0 = head + nvec * VEC;
    for (int part = 0; part < 2; ++part) {
        const int64_t i = part == 0 ? gtid : tail0 + gtid;
        if ((part == 0 && gtid < head) || (part == 1 && gtid < p.len - tail0)) {
            float acc = ld1<false>(src[0] + i);
#pragma unroll
            for (int r = 1; r < WT; ++r) acc = __fadd_rn(acc, ld1<false>(src[r] + i));
            if (p.do_scale) acc = __fmul_rn(acc, p.scale);
            if constexpr (MODE == kAllReduce) {
#pragma unroll
                for (int r = 0; r < WT; ++r) st1(const_cast<float *>(src[r]) + i, acc);
            } else {
                st1(p.out + i, acc);
            }
        }
    }
}

template <int WT, int MODE>
__global__ void __launch_bounds__(256) fold_table_fixed_kernel(const __grid_constant__ TableParams p)
{
    pdl_enter(p.pdl);
    const float *src[WT];
#pragma unroll
    for (int r = 0; r < WT; ++r) src[r] = p.table[r];
    int code = DETFOLD_OK;
#pragma unroll
    for (int r = 0; r < WT; ++r) {
        if (code == DETFOLD_OK && src[r] == nullptr) code = DETFOLD_ERR_NULL;
        if (code == DETFOLD_OK && ((uintptr_t)src[r] & 3u)) code = DETFOLD_ERR_ALIGN;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) *p.status = code;
    if (code != DETFOLD_OK) return;
    bool same8 = (MODE == kAllReduce) || phase_of(p.out, 8) == phase_of(src[0], 8);
    bool same4 = (MODE == kAllReduce) || phase_of(p.out, 4) == phase_of(src[0], 4);
#pragma unroll
    for (int r = 1; r < WT; ++r) {
        same8 = same8 && phase_of(src[r], 8) == phase_of(src[0], 8);
        same4 = same4 && phase_of(src[r], 4) == phase_of(src[0], 4);
    }
    if (same8) {
        int64_t head = (8 - phase_of(src[0], 8)) % 8;
        table_fixed_vec<WT, 8, MODE>(p, src, head > p.len ? p.len : head);
    } else if (same4) {
        int64_t head = (4 - phase_of(src[0], 4)) % 4;
        table_fixed_vec<WT, 4, MODE>(p, src, head > p.len ? p.len : head);
    } else {
        table_scalar_body<MODE>(p, src);
    }
}

template <int WT>
cudaError_t launch_table_fixed(const TableParams &p, int64_t work, bool small, int mode,
                               cudaStream_t stream)
{
    if (mode == kAllReduce)
        return launch_kernel<fold_table_fixed_kernel<WT, kAllReduce>>(p, work, 1, small, 256, 0, stream);
    return launch_kernel<fold_table_fixed_kernel<WT, kSumCoherent>>(p, work, 1, small, 256, 0, stream);
}

}  // namespace

cudaError_t launch_table(const float *const *d_table, float *out, int *d_status, int W, int64_t len,
                         float scale, int do_scale, int mode, cudaStream_t stream)
{
    TableParams p = {};
    p.table = d_table;
    p.out = out;
    p.status = d_status;
    p.len = len;
    p.scale = scale;
    p.do_scale = do_scale;
    p.W = W;
    const bool small = len <= DETFOLD_SMALL_LEN;
    p.pdl = ((small && DETFOLD_SMALL_PDL) || DETFOLD_PDL_ALL) ? 1 : 0;
    const int64_t work = (len + 7) / 8 > 0 ? (len + 7) / 8 : 1;  // vectors if 32-byte access
    // Small payloads: the register-table kernel (shortest dependent chain).
    // Bandwidth-sized calls: the shared-memory table kernel (fewer registers).
    switch (small ? W : 0) {
    case 1: return launch_table_fixed<1>(p, work, small, mode, stream);
    case 2: return launch_table_fixed<2>(p, work, small, mode, stream);
    case 3: return launch_table_fixed<3>(p, work, small, mode, stream);
    case 4: return launch_table_fixed<4>(p, work, small, mode, stream);
    case 5: return launch_table_fixed<5>(p, work, small, mode, stream);
    case 6: return launch_table_fixed<6>(p, work, small, mode, stream);
    case 7: return launch_table_fixed<7>(p, work, small, mode, stream);
    case 8: return launch_table_fixed<8>(p, work, small, mode, stream);
    default: break;
    }
    if (mode == kAllReduce)
        return launch_kernel<fold_table_kernel<kAllReduce>>(p, work, 1, small, 256, 0, stream);
    return launch_kernel<fold_table_kernel<kSumCoherent>>(p, work, 1, small, 256, 0, stream);
}

}  // namespace detfold
