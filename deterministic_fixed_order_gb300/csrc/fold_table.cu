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

// A small call at VEC-float width with a grid-stride loop (the 16-byte
// path of the small kernel below).
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

// The W entries of a small call, held in registers.
template <int WT>
struct SrcSet {
    const float *p[WT];
};

// Element i of a small call with scalar accesses (its head and tail).
template <int WT, int MODE>
__device__ __forceinline__ void table_fold_one(const TableParams &p, const SrcSet<WT> &s, int i)
{
    float acc = ld1<false>(s.p[0] + i);
#pragma unroll
    for (int r = 1; r < WT; ++r) acc = __fadd_rn(acc, ld1<false>(s.p[r] + i));
    if (p.do_scale) acc = __fmul_rn(acc, p.scale);
    if constexpr (MODE == kAllReduce) {
#pragma unroll
        for (int r = 0; r < WT; ++r) st1(const_cast<float *>(s.p[r]) + i, acc);
    } else {
        st1(p.out + i, acc);
    }
}

// Thread i < 8 folds head element i, thread 8 + j tail element j (inline,
// as the fold's own small kernel does).
template <int WT, int MODE>
__device__ __forceinline__ void table_small_edges(const TableParams &p, SrcSet<WT> s, int i, int head, int tail0)
{
    if (i < 8 ? i < head : i - 8 < (int)p.len - tail0)
        table_fold_one<WT, MODE>(p, s, i < 8 ? i : tail0 + (i - 8));
}

// A small call whose entries share no 32-byte phase: 16-byte vectors if
// they share a 16-byte phase, else scalars.
template <int WT, int MODE>
__device__ __noinline__ void table_small_slow(const TableParams &p, SrcSet<WT> s, bool same4)
{
    if (same4) {
        const int64_t head = (4 - phase_of(s.p[0], 4)) % 4;
        table_fixed_vec<WT, 4, MODE>(p, s.p, head > p.len ? p.len : head);
    } else {
        table_scalar_body<MODE>(p, s.p);
    }
}

// Small payloads (len <= DETFOLD_SMALL_LEN) with W <= 8. Every thread reads
// the (broadcast) table entries into registers and checks them itself, with
// no shared memory and no block barrier between the table load and the data
// loads. The common case, every entry (and the output) at one 32-byte phase,
// is one 32-byte vector per thread with 32-bit indices; the head and tail
// run in a leading CTA of their own and the narrower widths out of line, so
// the code a CTA executes after the wait -- what the latency of a graph of
// small folds is made of -- stays short.
template <int WT, int MODE>
__global__ void __launch_bounds__(DETFOLD_SMALL_THREADS) fold_table_small_kernel(const __grid_constant__ TableParams p)
{
    static_assert(DETFOLD_SMALL_LEN < (1 << 30), "small-path indices are 32-bit");
    pdl_enter(p.pdl);
    SrcSet<WT> s;
#pragma unroll
    for (int r = 0; r < WT; ++r) s.p[r] = p.table[r];
    int code = DETFOLD_OK;
#pragma unroll
    for (int r = 0; r < WT; ++r) {
        if (code == DETFOLD_OK && s.p[r] == nullptr) code = DETFOLD_ERR_NULL;
        if (code == DETFOLD_OK && ((uintptr_t)s.p[r] & 3u)) code = DETFOLD_ERR_ALIGN;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) *p.status = code;
    if (code != DETFOLD_OK) return;
    // byte phase within 32 bytes; every pointer is 4-byte aligned here
    const unsigned ph0 = (unsigned)(uintptr_t)s.p[0] & 31u;
    unsigned diff = (MODE == kAllReduce) ? 0u : (((unsigned)(uintptr_t)p.out & 31u) ^ ph0);
#pragma unroll
    for (int r = 1; r < WT; ++r) diff |= ((unsigned)(uintptr_t)s.p[r] & 31u) ^ ph0;
    if (diff != 0) {
        table_small_slow<WT, MODE>(p, s, (diff & 15u) == 0);
        return;
    }
    const int len = (int)p.len;
    int head = (int)(((32u - ph0) & 31u) / 4);
    if (head > len) head = len;
    const int nvec = (len - head) / 8;
    const int tail0 = head + nvec * 8;
    // the first CTA folds the head and the tail alone (the host always adds
    // it: only the device sees the entries' phases), so their memory round
    // trip runs beside the vectors' instead of after one thread's vector
    if (blockIdx.x == 0) {
        if ((head != 0 || tail0 != len) && threadIdx.x < 16)
            table_small_edges<WT, MODE>(p, s, threadIdx.x, head, tail0);
        return;
    }
    const int i = (blockIdx.x - 1) * blockDim.x + threadIdx.x;
    if (i < nvec) {
        const int e = head + i * 8;
        Vec<8> x[WT];
#pragma unroll
        for (int r = 0; r < WT; ++r) x[r] = ldv<8, false>(s.p[r] + e);
        Vec<8> acc = x[0];
#pragma unroll
        for (int r = 1; r < WT; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc.v[j] = __fadd_rn(acc.v[j], x[r].v[j]);
        if (p.do_scale) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc.v[j] = __fmul_rn(acc.v[j], p.scale);
        }
        if constexpr (MODE == kAllReduce) {
#pragma unroll
            for (int r = 0; r < WT; ++r) stv<8>(const_cast<float *>(s.p[r]) + e, acc);
        } else {
            stv<8>(p.out + e, acc);
        }
    }
}

template <int WT>
cudaError_t launch_table_small(const TableParams &p, int64_t work, int mode, cudaStream_t stream)
{
    // one leading CTA for the edges (fold_table_small_kernel)
    if (mode == kAllReduce)
        return launch_kernel<fold_table_small_kernel<WT, kAllReduce>>(p, work, 1, true, 256, 0, stream, true, 1);
    return launch_kernel<fold_table_small_kernel<WT, kSumCoherent>>(p, work, 1, true, 256, 0, stream, true, 1);
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
    // Bulk-sized calls with W <= 8: the bulk-async pipeline, fed from the table.
    if (DETFOLD_USE_BULK && !small && W <= 8 && len >= DETFOLD_BULK_TABLE_MIN_LEN)
        return launch_bulk_table(d_table, out, d_status, W, len, scale, do_scale, mode, stream);
    // Small payloads: the register-table kernel (shortest dependent chain;
    // one thread per 32-byte vector). Bandwidth-sized calls: the
    // shared-memory table kernel (fewer registers).
    switch (small ? W : 0) {
    case 1: return launch_table_small<1>(p, work, mode, stream);
    case 2: return launch_table_small<2>(p, work, mode, stream);
    case 3: return launch_table_small<3>(p, work, mode, stream);
    case 4: return launch_table_small<4>(p, work, mode, stream);
    case 5: return launch_table_small<5>(p, work, mode, stream);
    case 6: return launch_table_small<6>(p, work, mode, stream);
    case 7: return launch_table_small<7>(p, work, mode, stream);
    case 8: return launch_table_small<8>(p, work, mode, stream);
    default: break;
    }
    if (mode == kAllReduce)
        return launch_kernel<fold_table_kernel<kAllReduce>>(p, work, 1, small, 256, 0, stream);
    return launch_kernel<fold_table_kernel<kSumCoherent>>(p, work, 1, small, 256, 0, stream);
}

}  // namespace detfold
