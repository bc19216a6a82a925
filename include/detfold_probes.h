/*
 * libdetfold_probes -- measurement probes for libdetfold (not part of the
 * fold library's ABI, and not loaded by its Python binding).
 *
 * The pages have no counterpart. The fold's latency target for small payloads
 * (the 16 KiB decode join of memra-engine 0.128.0 tests/tp_ar_gpu.rs, module
 * note) is "the launch-latency floor"; these kernels measure that floor on
 * the same GPU, in the same way the small folds are launched: back to back on
 * one stream (normally captured in a CUDA graph), with programmatic dependent
 * launch, each launch's loads issued only after the preceding grid retired.
 *
 * Return value: DETFOLD_OK (0) or a negative DETFOLD_ERR_* code of detfold.h
 * (nothing is enqueued on an argument error; DETFOLD_ERR_CUDA after a failed
 * launch, with the cudaError_t value kept for detfold_probe_last_cuda_error).
 * `stream` is a cudaStream_t passed as void*. Nothing allocates or synchronizes.
 */
#ifndef DETFOLD_PROBES_H
#define DETFOLD_PROBES_H

#include <stdint.h>

#include "detfold.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest n of detfold_probe_same_shape_floor (the small-payload limit). */
#define DETFOLD_PROBE_SAME_SHAPE_MAX_N (1 << 17)
/* n of detfold_probe_same_shape_floor must be a multiple of this: one 32-byte
 * vector per thread, 128-thread CTAs, an exact grid. */
#define DETFOLD_PROBE_SAME_SHAPE_QUANTUM 1024

/*
 * `count` launches of an empty kernel (one CTA of 32 threads), with
 * programmatic dependent launch when pdl != 0. count < 0 -> ERR_ARG.
 */
DETFOLD_API int detfold_probe_launch_floor(int count, int pdl, void *stream);

/*
 * `count` launches of a one-warp kernel in which lane t copies src[t] to
 * dst[t] (t < 32), the load issued after the preceding grid retired. The
 * least that any launch takes which reads what a predecessor may have
 * written and writes its own result.
 *   src, dst  device, 32 floats each, 4-byte aligned, disjoint.
 * NULL -> ERR_NULL; count < 0 -> ERR_ARG; misaligned -> ERR_ALIGN;
 * overlap -> ERR_OVERLAP.
 */
DETFOLD_API int detfold_probe_memory_floor(const float *src, float *dst, int count, int pdl, void *stream);

/*
 * `count` launches shaped exactly as the W=2 small-payload fold of n floats
 * when its operands sit on one 32-byte phase: n/1024 CTAs of 128 threads,
 * one thread per 32-byte vector, programmatic dependent launch, both sources
 * loaded through the read-only path after the wait, one 32-byte store --
 * but no adds: out[i] = src0[i] for even i and src1[i] for odd i. A graph of
 * these is the floor of a graph of 16 KiB W=2 folds that moves the same
 * bytes with the same launch shape.
 *   out, src0, src1  device, n floats each, 32-byte aligned; out disjoint
 *                    from both sources (sources may overlap each other).
 *   n                1024 <= n <= DETFOLD_PROBE_SAME_SHAPE_MAX_N, a multiple
 *                    of DETFOLD_PROBE_SAME_SHAPE_QUANTUM (else ERR_LEN).
 * NULL -> ERR_NULL; count < 0 -> ERR_ARG; not 32-byte aligned -> ERR_ALIGN;
 * overlap -> ERR_OVERLAP.
 */
DETFOLD_API int detfold_probe_same_shape_floor(float *out, const float *src0, const float *src1, int64_t n,
                                               int count, void *stream);

/* The cudaError_t value of the last DETFOLD_ERR_CUDA returned by a probe on
 * the calling thread (0 if none). */
DETFOLD_API int detfold_probe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DETFOLD_PROBES_H */
