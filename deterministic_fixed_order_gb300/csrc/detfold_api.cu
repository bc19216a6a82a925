// The C ABI of libdetfold (declared in include/detfold.h): argument
// validation, the shard plan, dispatch to the fold and movement launchers,
// and the staged comparator's schedule. Nothing here allocates, synchronizes or
// touches device memory other than through stream-ordered launches and
// copies.
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "detfold.h"
#include "detfold_launch.cuh"

namespace detfold {
// One-shot all-reduce emulation, one cooperative launch (one_shot.cu).
cudaError_t launch_one_shot(float *const *arenas, int W, int64_t len, float scale, int do_scale,
                            void *link, unsigned long long epoch, float *stage, int *words,
                            long long wait_ns, int drop_rank, int drop_at_exit,
                            cudaStream_t stream);
}  // namespace detfold

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return DETFOLD_OK;
    g_last_cuda_error = (int)e;
    (void)cudaGetLastError();  // clear a non-sticky launch error
    return DETFOLD_ERR_CUDA;
}

bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) intersect.
bool intersects(const void *a, int64_t na, const void *b, int64_t nb)
{
    const uintptr_t ua = (uintptr_t)a, ub = (uintptr_t)b;
    return ua < ub + (uintptr_t)nb && ub < ua + (uintptr_t)na;
}

int check_world(int W) { return (W < 1 || W > DETFOLD_MAX_W) ? DETFOLD_ERR_WORLD : DETFOLD_OK; }

int check_len(int64_t len) { return (len < 0 || len > DETFOLD_MAX_LEN) ? DETFOLD_ERR_LEN : DETFOLD_OK; }

void plan_shards(int64_t len, int W, int64_t *starts, int64_t *lens)
{
    const int64_t base = len / W, rem = len % W;
    for (int r = 0; r < W; ++r) {
        starts[r] = (int64_t)r * base + (r < rem ? r : rem);
        lens[r] = base + (r < rem ? 1 : 0);
    }
}

// Stack row stride (elements) of the staged comparator: the largest shard
// plus room to shift a row by up to 7 elements, rounded to 64 elements.
int64_t staged_row_stride(int64_t len, int W)
{
    const int64_t max_shard = (len + W - 1) / W;
    return (max_shard + 8 + 63) / 64 * 64;
}

cudaError_t launch(const detfold::LaunchSpec &s, cudaStream_t st)
{
    switch (s.mode) {
    case detfold::kSumNC: return detfold::launch_sum_nc(s, st);
    case detfold::kSumCoherent: return detfold::launch_sum_coherent(s, st);
    default: return detfold::launch_allreduce(s, st);
    }
}

int arenas_valid(float *const *arenas, int W, int64_t len)
{
    if (!arenas) return DETFOLD_ERR_NULL;
    for (int r = 0; r < W; ++r)
        if (!arenas[r]) return DETFOLD_ERR_NULL;
    for (int r = 0; r < W; ++r)
        if (!aligned4(arenas[r])) return DETFOLD_ERR_ALIGN;
    const int64_t bytes = len * 4;
    for (int a = 0; a < W; ++a)
        for (int b = a + 1; b < W; ++b)
            if (arenas[a] == arenas[b] || intersects(arenas[a], bytes, arenas[b], bytes))
                return DETFOLD_ERR_OVERLAP;
    return DETFOLD_OK;
}

}  // namespace

namespace detfold {

// Records a failed CUDA call for detfold_last_cuda_error (for entry points
// defined in other translation units).
int record_cuda_status(cudaError_t e) { return cuda_status(e); }

}  // namespace detfold

extern "C" {

int detfold_sum_stacked(float *out, const float *stacked, int W, int64_t len, void *stream)
{
    if (!out || !stacked) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    if (!aligned4(out) || !aligned4(stacked)) return DETFOLD_ERR_ALIGN;
    if (len == 0) return DETFOLD_OK;
    if (intersects(out, len * 4, stacked, (int64_t)W * len * 4)) return DETFOLD_ERR_OVERLAP;
    const float *rows[DETFOLD_MAX_W];
    for (int r = 0; r < W; ++r) rows[r] = stacked + (int64_t)r * len;
    detfold::LaunchSpec s = {W, detfold::kSumNC, rows, out, len, 1.0f, 0};
    return cuda_status(launch(s, (cudaStream_t)stream));
}

int detfold_sum_ptrs(float *out, const float *const *srcs, int W, int64_t len, void *stream)
{
    if (!out || !srcs) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    for (int r = 0; r < W; ++r)
        if (!srcs[r]) return DETFOLD_ERR_NULL;
    if (int rc = check_len(len)) return rc;
    if (!aligned4(out)) return DETFOLD_ERR_ALIGN;
    for (int r = 0; r < W; ++r)
        if (!aligned4(srcs[r])) return DETFOLD_ERR_ALIGN;
    if (len == 0) return DETFOLD_OK;
    bool in_place = false;
    for (int r = 0; r < W; ++r) {
        if (srcs[r] == out) {
            in_place = true;
        } else if (intersects(out, len * 4, srcs[r], len * 4)) {
            return DETFOLD_ERR_OVERLAP;
        }
    }
    if (W == 1 && in_place) return DETFOLD_OK;  // the fold of one addend is itself
    detfold::LaunchSpec s = {W, in_place ? detfold::kSumCoherent : detfold::kSumNC, srcs, out, len,
                             1.0f, 0};
    return cuda_status(launch(s, (cudaStream_t)stream));
}

int detfold_scale(float *buf, int64_t len, float scale, void *stream)
{
    if (!buf) return DETFOLD_ERR_NULL;
    if (int rc = check_len(len)) return rc;
    if (!aligned4(buf)) return DETFOLD_ERR_ALIGN;
    if (len == 0 || scale == 1.0f) return DETFOLD_OK;
    const float *one[1] = {buf};
    detfold::LaunchSpec s = {1, detfold::kAllReduce, one, nullptr, len, scale, 1};
    return cuda_status(launch(s, (cudaStream_t)stream));
}

int detfold_loopback_allreduce(float *const *arenas, int W, int64_t len, float mean_scale,
                               void *stream)
{
    if (!arenas) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    if (int rc = arenas_valid(arenas, W, len)) return rc;
    if (len == 0) return DETFOLD_OK;
    const int do_scale = mean_scale != 1.0f;
    if (W == 1 && !do_scale) return DETFOLD_OK;
    detfold::LaunchSpec s = {W, detfold::kAllReduce, (const float *const *)arenas, nullptr, len,
                             mean_scale, do_scale};
    return cuda_status(launch(s, (cudaStream_t)stream));
}

int64_t detfold_staged_workspace_bytes(int64_t len, int W)
{
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    return ((int64_t)W * staged_row_stride(len, W) + 8) * 4;
}

int detfold_mean_scale(int W, float *scale)
{
    if (!scale) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    // one IEEE binary32 division, rounded to nearest-even (host SSE / NEON)
    volatile float w = (float)W;  // W <= 256 converts exactly
    *scale = 1.0f / w;
    return DETFOLD_OK;
}

int detfold_loopback_allreduce_staged(float *const *arenas, int W, int64_t len, float mean_scale,
                                      void *workspace, int64_t workspace_bytes, void *stream)
{
    return detfold_loopback_allreduce_staged_ex(arenas, W, len, mean_scale, 0, workspace,
                                                workspace_bytes, stream);
}

int detfold_loopback_allreduce_staged_ex(float *const *arenas, int W, int64_t len, float mean_scale,
                                         int flags, void *workspace, int64_t workspace_bytes,
                                         void *stream)
{
    if (!arenas) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    if (flags & ~(DETFOLD_STAGED_REVERSE_DELIVERY | DETFOLD_STAGED_SEPARATE_SCALE |
                  DETFOLD_STAGED_CE_COPIES))
        return DETFOLD_ERR_ARG;
    if (int rc = arenas_valid(arenas, W, len)) return rc;
    const bool do_scale = mean_scale != 1.0f;
    if (len == 0) return DETFOLD_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (W == 1) {
        // The reference's round is a no-op for one rank; only the mean remains.
        return detfold_scale(arenas[0], len, mean_scale, stream);
    }
    const int64_t need = detfold_staged_workspace_bytes(len, W);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15u))
        return DETFOLD_ERR_WORKSPACE;
    for (int r = 0; r < W; ++r)
        if (intersects(workspace, workspace_bytes, arenas[r], len * 4)) return DETFOLD_ERR_OVERLAP;

    int64_t starts[DETFOLD_MAX_W], lens[DETFOLD_MAX_W];
    plan_shards(len, W, starts, lens);
    const int64_t stride = staged_row_stride(len, W);
    float *ws = (float *)(((uintptr_t)workspace + 31u) & ~(uintptr_t)31u);
    const bool reverse = flags & DETFOLD_STAGED_REVERSE_DELIVERY;
    const bool separate = flags & DETFOLD_STAGED_SEPARATE_SCALE;

    const bool ce = flags & DETFOLD_STAGED_CE_COPIES;

    // Phase A: per owner, exchange into slot = source rank, then fold.
    for (int o = 0; o < W; ++o) {
        const int64_t n = lens[o], s0 = starts[o];
        if (n == 0) continue;
        float *dst = arenas[o] + s0;
        const int ph = detfold::elem_phase(dst, 8);  // rows share the shard's 32-byte phase
        const float *rows[DETFOLD_MAX_W];
        for (int r = 0; r < W; ++r) rows[r] = ws + (int64_t)r * stride + ph;
        const float *from[DETFOLD_MAX_W];
        float *to[DETFOLD_MAX_W];
        for (int k = 0; k < W; ++k) {
            const int src = reverse ? W - 1 - k : k;
            from[k] = arenas[src] + s0;
            to[k] = const_cast<float *>(rows[src]);
        }
        if (ce) {
            for (int k = 0; k < W; ++k) {
                cudaError_t e = cudaMemcpyAsync(to[k], from[k], (size_t)n * 4,
                                                cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return cuda_status(e);
            }
        } else if (int rc = cuda_status(detfold::launch_move(from, to, W, n, st))) {
            return rc;
        }
        detfold::LaunchSpec s = {W, detfold::kSumNC, rows, dst, n, mean_scale,
                                 (do_scale && !separate) ? 1 : 0};
        if (int rc = cuda_status(launch(s, st))) return rc;
        if (do_scale && separate) {
            if (int rc = detfold_scale(dst, n, mean_scale, stream)) return rc;
        }
    }
    // Phase B: every owner's shard to every other arena.
    for (int o = 0; o < W; ++o) {
        const int64_t n = lens[o], s0 = starts[o];
        if (n == 0) continue;
        const float *from[DETFOLD_MAX_W];
        float *to[DETFOLD_MAX_W];
        int K = 0;
        for (int r = 0; r < W; ++r) {
            if (r == o) continue;
            from[K] = arenas[o] + s0;
            to[K++] = arenas[r] + s0;
        }
        if (ce) {
            for (int k = 0; k < K; ++k) {
                cudaError_t e = cudaMemcpyAsync(to[k], from[k], (size_t)n * 4,
                                                cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return cuda_status(e);
            }
        } else if (int rc = cuda_status(detfold::launch_move(from, to, K, n, st))) {
            return rc;
        }
    }
    return DETFOLD_OK;
}

int detfold_broadcast(float *const *dsts, int ndst, const float *src, int64_t len, void *stream)
{
    if (!dsts || !src) return DETFOLD_ERR_NULL;
    if (int rc = check_world(ndst)) return rc;
    for (int k = 0; k < ndst; ++k)
        if (!dsts[k]) return DETFOLD_ERR_NULL;
    if (int rc = check_len(len)) return rc;
    if (!aligned4(src)) return DETFOLD_ERR_ALIGN;
    if (int rc = arenas_valid(dsts, ndst, len)) return rc;
    if (len == 0) return DETFOLD_OK;
    for (int k = 0; k < ndst; ++k)
        if (intersects(dsts[k], len * 4, src, len * 4)) return DETFOLD_ERR_OVERLAP;
    const float *from[DETFOLD_MAX_W];
    for (int k = 0; k < ndst; ++k) from[k] = src;
    return cuda_status(detfold::launch_move(from, dsts, ndst, len, (cudaStream_t)stream));
}

int detfold_all_gather(float *const *outs, int W, const float *const *parts, int64_t span,
                       void *stream)
{
    if (!outs || !parts) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    for (int r = 0; r < W; ++r)
        if (!outs[r] || !parts[r]) return DETFOLD_ERR_NULL;
    if (int rc = check_len(span)) return rc;
    if ((int64_t)W * span > DETFOLD_MAX_LEN) return DETFOLD_ERR_LEN;
    for (int r = 0; r < W; ++r)
        if (!aligned4(parts[r])) return DETFOLD_ERR_ALIGN;
    const int64_t total = (int64_t)W * span;
    if (int rc = arenas_valid(outs, W, total)) return rc;
    if (span == 0) return DETFOLD_OK;
    for (int r = 0; r < W; ++r)
        for (int p = 0; p < W; ++p)
            if (intersects(outs[r], total * 4, parts[p], span * 4)) return DETFOLD_ERR_OVERLAP;
    // Part p lands at offset p*span of every output. With at most 8 parts and
    // every pair at one 16-byte phase, all W*W pairs go in one launch, ordered
    // by part (the bulk movement path reads each part once and stores it W
    // times); otherwise one broadcast per part.
    if (W <= 8) {
        const uintptr_t ph = (uintptr_t)parts[0] & 15u;
        bool same = true;
        for (int p = 0; same && p < W; ++p) {
            same = ((uintptr_t)parts[p] & 15u) == ph;
            for (int r = 0; same && r < W; ++r) same = ((uintptr_t)(outs[r] + (int64_t)p * span) & 15u) == ph;
        }
        if (same) {
            const float *from[64];
            float *to[64];
            for (int p = 0; p < W; ++p)
                for (int r = 0; r < W; ++r) {
                    from[p * W + r] = parts[p];
                    to[p * W + r] = outs[r] + (int64_t)p * span;
                }
            return cuda_status(detfold::launch_move(from, to, W * W, span, (cudaStream_t)stream));
        }
    }
    for (int p = 0; p < W; ++p) {
        const float *from[DETFOLD_MAX_W];
        float *to[DETFOLD_MAX_W];
        for (int r = 0; r < W; ++r) {
            from[r] = parts[p];
            to[r] = outs[r] + (int64_t)p * span;
        }
        if (int rc = cuda_status(detfold::launch_move(from, to, W, span, (cudaStream_t)stream)))
            return rc;
    }
    return DETFOLD_OK;
}

int detfold_sum_ptrs_dev(float *out, const float *const *d_srcs, int W, int64_t len, int *d_status,
                         void *stream)
{
    if (!out || !d_srcs) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    if (!aligned4(out) || ((uintptr_t)d_srcs & 7u) || ((uintptr_t)d_status & 3u))
        return DETFOLD_ERR_ALIGN;
    if (len == 0) return DETFOLD_OK;
    return cuda_status(detfold::launch_table(d_srcs, out, d_status, W, len, 1.0f, 0,
                                             detfold::kSumCoherent, (cudaStream_t)stream));
}

int detfold_loopback_allreduce_dev(float *const *d_arenas, int W, int64_t len, float mean_scale,
                                   int *d_status, void *stream)
{
    if (!d_arenas) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    if (((uintptr_t)d_arenas & 7u) || ((uintptr_t)d_status & 3u)) return DETFOLD_ERR_ALIGN;
    const int do_scale = mean_scale != 1.0f;
    if (len == 0 || (W == 1 && !do_scale)) return DETFOLD_OK;
    return cuda_status(detfold::launch_table((const float *const *)d_arenas, nullptr, d_status, W,
                                             len, mean_scale, do_scale, detfold::kAllReduce,
                                             (cudaStream_t)stream));
}

int detfold_one_shot_allreduce(float *const *arenas, int W, int64_t len, float mean_scale,
                               void *link, uint64_t epoch, float *stage, int *words,
                               int64_t wait_ns, int drop_rank, int drop_at_exit, void *stream)
{
    if (!arenas || !link || !stage || !words) return DETFOLD_ERR_NULL;
    if (W < 1 || W > DETFOLD_ONESHOT_MAX_W) return DETFOLD_ERR_WORLD;
    if (len < 0 || len > DETFOLD_ONESHOT_MAX_LEN) return DETFOLD_ERR_LEN;
    if (wait_ns < 1 || wait_ns > 2000000000LL || drop_rank < -1 || drop_rank >= W)
        return DETFOLD_ERR_ARG;
    if (((uintptr_t)link & 7u) || !aligned4(stage) || ((uintptr_t)words & 3u))
        return DETFOLD_ERR_ALIGN;
    if (int rc = arenas_valid(arenas, W, len)) return rc;
    if (len == 0) return DETFOLD_OK;
    const int64_t stage_bytes = (int64_t)W * len * 4;
    for (int r = 0; r < W; ++r)
        if (intersects(stage, stage_bytes, arenas[r], len * 4) ||
            intersects(link, DETFOLD_ONESHOT_LINK_BYTES, arenas[r], len * 4))
            return DETFOLD_ERR_OVERLAP;
    if (intersects(stage, stage_bytes, link, DETFOLD_ONESHOT_LINK_BYTES)) return DETFOLD_ERR_OVERLAP;
    return cuda_status(detfold::launch_one_shot(arenas, W, len, mean_scale, mean_scale != 1.0f ? 1 : 0,
                                                link, epoch, stage, words, wait_ns, drop_rank,
                                                drop_at_exit ? 1 : 0, (cudaStream_t)stream));
}

int detfold_shard_plan(int64_t len, int W, int64_t *starts, int64_t *lens)
{
    if (!starts || !lens) return DETFOLD_ERR_NULL;
    if (int rc = check_world(W)) return rc;
    if (int rc = check_len(len)) return rc;
    plan_shards(len, W, starts, lens);
    return DETFOLD_OK;
}

const char *detfold_status_string(int status)
{
    switch (status) {
    case DETFOLD_OK: return "ok";
    case DETFOLD_ERR_NULL: return "a required pointer is NULL";
    case DETFOLD_ERR_WORLD: return "W is outside [1, DETFOLD_MAX_W]";
    case DETFOLD_ERR_LEN: return "len is negative or above DETFOLD_MAX_LEN";
    case DETFOLD_ERR_ALIGN: return "a device pointer is not 4-byte aligned";
    case DETFOLD_ERR_OVERLAP: return "operands overlap in a way this call forbids";
    case DETFOLD_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case DETFOLD_ERR_CUDA: return "a CUDA call failed (see detfold_last_cuda_error)";
    case DETFOLD_ERR_ARG: return "invalid argument";
    case DETFOLD_ERR_SCRATCH_LIMIT:
        return "request needs more than the library's static scratch (DETFOLD_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
    }
}

int detfold_last_cuda_error(void) { return g_last_cuda_error; }

int detfold_pipeline_timeouts(int64_t *count)
{
    if (!count) return DETFOLD_ERR_NULL;
    unsigned long long a = 0, b = 0;
    if (int rc = cuda_status(detfold::read_pipeline_timeouts_bulk(&a))) return rc;
    if (int rc = cuda_status(detfold::read_pipeline_timeouts_move(&b))) return rc;
    *count = (int64_t)(a + b);
    return DETFOLD_OK;
}

}  // extern "C"
