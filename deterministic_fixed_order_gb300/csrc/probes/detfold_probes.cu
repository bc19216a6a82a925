// Measurement probes (include/detfold_probes.h): the floors that graphs of
// small folds are measured against. Built as their own library,
// libdetfold_probes.so; the fold library neither contains nor loads them.
//
// Every probe launches the way the small-payload folds launch: a
// cudaLaunchKernelEx on the caller's stream with programmatic dependent
// launch when asked, `griddepcontrol.wait` before the first load and
// `launch_dependents` right after it.
#include <cstdint>
#include <cuda_runtime.h>

#include "detfold_kernels.cuh"
#include "detfold_probes.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return DETFOLD_OK;
    g_last_cuda_error = (int)e;
    (void)cudaGetLastError();
    return DETFOLD_ERR_CUDA;
}

bool intersects(const void *a, int64_t na, const void *b, int64_t nb)
{
    const uintptr_t ua = (uintptr_t)a, ub = (uintptr_t)b;
    return ua < ub + (uintptr_t)nb && ub < ua + (uintptr_t)na;
}

__global__ void empty_kernel(int pdl) { detfold::pdl_enter(pdl); }

// One warp: each lane copies one float, loaded only after the preceding
// grid has retired.
__global__ void copy_warp_kernel(const float *__restrict__ src, float *__restrict__ dst, int pdl)
{
    detfold::pdl_enter(pdl);
    dst[threadIdx.x] = src[threadIdx.x];
}

// The W=2 small-path fold's body without its adds: the same two read-only
// 32-byte loads per thread and the same 32-byte store (even lanes of the
// vector from src0, odd ones from src1, so both loads feed the store).
__global__ void __launch_bounds__(128) same_shape_kernel(const float *src0, const float *src1, float *out)
{
    detfold::pdl_enter(1);
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
    const detfold::Vec<8> a = detfold::ldv<8, true>(src0 + e);
    const detfold::Vec<8> b = detfold::ldv<8, true>(src1 + e);
    detfold::Vec<8> o;
#pragma unroll
    for (int k = 0; k < 8; ++k) o.v[k] = (k & 1) ? b.v[k] : a.v[k];
    detfold::stv<8>(out + e, o);
}

template <typename... Params, typename... Args>
cudaError_t launch_n(void (*kernel)(Params...), int count, int grid, int threads, int pdl,
                     cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    for (int k = 0; k < count; ++k) {
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

int detfold_probe_launch_floor(int count, int pdl, void *stream)
{
    if (count < 0) return DETFOLD_ERR_ARG;
    pdl = pdl ? 1 : 0;
    return cuda_status(launch_n(empty_kernel, count, 1, 32, pdl, (cudaStream_t)stream, pdl));
}

int detfold_probe_memory_floor(const float *src, float *dst, int count, int pdl, void *stream)
{
    if (!src || !dst) return DETFOLD_ERR_NULL;
    if (count < 0) return DETFOLD_ERR_ARG;
    if (((uintptr_t)src & 3u) || ((uintptr_t)dst & 3u)) return DETFOLD_ERR_ALIGN;
    if (intersects(src, 32 * sizeof(float), dst, 32 * sizeof(float))) return DETFOLD_ERR_OVERLAP;
    pdl = pdl ? 1 : 0;
    return cuda_status(launch_n(copy_warp_kernel, count, 1, 32, pdl, (cudaStream_t)stream, src, dst, pdl));
}

int detfold_probe_same_shape_floor(float *out, const float *src0, const float *src1, int64_t n, int count,
                                   void *stream)
{
    if (!out || !src0 || !src1) return DETFOLD_ERR_NULL;
    if (count < 0) return DETFOLD_ERR_ARG;
    if (n < DETFOLD_PROBE_SAME_SHAPE_QUANTUM || n > DETFOLD_PROBE_SAME_SHAPE_MAX_N ||
        n % DETFOLD_PROBE_SAME_SHAPE_QUANTUM)
        return DETFOLD_ERR_LEN;
    if (((uintptr_t)out & 31u) || ((uintptr_t)src0 & 31u) || ((uintptr_t)src1 & 31u)) return DETFOLD_ERR_ALIGN;
    if (intersects(out, n * 4, src0, n * 4) || intersects(out, n * 4, src1, n * 4)) return DETFOLD_ERR_OVERLAP;
    const int grid = (int)(n / DETFOLD_PROBE_SAME_SHAPE_QUANTUM);
    return cuda_status(launch_n(same_shape_kernel, count, grid, 128, 1, (cudaStream_t)stream, src0, src1, out));
}

int detfold_probe_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
