/*
 * libdetfold -- fixed-order elementwise fold for GB300 (sm_103a).
 *
 * What is computed (mamba-rs 0.6.2 src/dist/reducer.rs, module doc and
 * `reduce_sum_reference`): for W rank addends s_0..s_{W-1} of an f32 arena,
 *
 *     out[i] = ((s_0[i] + s_1[i]) + s_2[i]) + ... + s_{W-1}[i]
 *
 * a serial IEEE binary32 round-to-nearest-even add chain in strictly
 * ascending source-rank order, starting from s_0[i] (so an all -0 column
 * stays -0). Subnormals are kept (no flush to zero). The bits therefore do
 * not depend on the launch shape, the transport or the delivery order. The
 * optional mean is a separate multiply, out[i] = fl(sum[i] * mean_scale),
 * with mean_scale normally fl(1/W), which is exact for power-of-two W
 * unless the product underflows.
 *
 * Conventions shared by every entry point:
 *   - Return value: DETFOLD_OK (0) or a negative DETFOLD_ERR_* code. No
 *     entry point aborts, prints or allocates device memory, and none
 *     synchronizes except the diagnostic detfold_pipeline_timeouts.
 *     On any error nothing has been enqueued, except DETFOLD_ERR_CUDA from
 *     a multi-launch call, where earlier launches may already be enqueued.
 *   - Pointers named "device" are caller-owned device memory of the current
 *     device (for example torch tensors); the library keeps no reference
 *     after the call returns. They must be 4-byte aligned; any 4-byte
 *     phase is legal (vector loads are used where every operand shares
 *     the same 16- or 32-byte phase, scalar loads otherwise).
 *   - Arrays named "host" (pointer tables, shard-plan outputs) are read or
 *     written only during the call. Pointer tables are copied into kernel
 *     parameters, so a captured CUDA graph keeps the addresses it saw.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). All device work is stream-ordered and asynchronous.
 *   - len is an element count (f32 words); len == 0 is a no-op returning
 *     DETFOLD_OK once the pointer and W arguments have been checked
 *     (mamba-rs src/dist/reducer.rs `DetReduceKernel::launch`, `copy_d2d`).
 *   - W (the world size) must be 1 <= W <= DETFOLD_MAX_W
 *     (`reduce_sum_reference` asserts a non-empty world).
 *   - Per device, the library caches what it looks up once: kernel
 *     attributes, resident-CTA counts and the address of its static scratch
 *     array. Do not reset a device (cudaDeviceReset) or otherwise replace its
 *     primary context while the library is in use in the process: later
 *     calls would use the cached values of the old context.
 */
#ifndef DETFOLD_H
#define DETFOLD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility; only the entry points
 * declared here are exported. */
#if defined(__GNUC__)
#define DETFOLD_API __attribute__((visibility("default")))
#else
#define DETFOLD_API
#endif

#define DETFOLD_MAX_W 256
/* Largest accepted len: 2^40 elements (4 TiB per addend). */
#define DETFOLD_MAX_LEN ((int64_t)1 << 40)

/* Status codes. */
#define DETFOLD_OK 0
#define DETFOLD_ERR_NULL (-1)      /* a required pointer is NULL                    */
#define DETFOLD_ERR_WORLD (-2)     /* W < 1 or W > DETFOLD_MAX_W                    */
#define DETFOLD_ERR_LEN (-3)       /* len < 0 or len > DETFOLD_MAX_LEN               */
#define DETFOLD_ERR_ALIGN (-4)     /* a device pointer is not 4-byte aligned         */
#define DETFOLD_ERR_OVERLAP (-5)   /* operands overlap in a way the call forbids     */
#define DETFOLD_ERR_WORKSPACE (-6) /* workspace missing, too small or misaligned     */
#define DETFOLD_ERR_CUDA (-7)      /* a CUDA call failed; see detfold_last_cuda_error */
#define DETFOLD_ERR_ARG (-8)       /* another invalid argument (unknown flag bits)   */
#define DETFOLD_ERR_SCRATCH_LIMIT (-9) /* request needs more than the static scratch  */

/* Flags of detfold_loopback_allreduce_staged_ex. */
#define DETFOLD_STAGED_REVERSE_DELIVERY 1 /* copy peers into the stack in descending rank order */
#define DETFOLD_STAGED_SEPARATE_SCALE 2   /* mean multiply as its own pass, not in the fold store */
#define DETFOLD_STAGED_CE_COPIES 4        /* move bytes with cudaMemcpyAsync (copy engines), as the
                                             reference's copy_d2d does, instead of the SM movement kernel */

/*
 * Stacked fold (mamba-rs src/dist/reducer.rs, `DET_SUM_RANKS_SRC` and
 * `DetReduceKernel::launch`).
 *   out     device, len f32, written.
 *   stacked device, row-major [W][len] f32, slot (row) r = source rank r, read.
 *   out must not overlap stacked (DETFOLD_ERR_OVERLAP).
 * W == 1 copies row 0 into out.
 */
DETFOLD_API int detfold_sum_stacked(float *out, const float *stacked, int W, int64_t len, void *stream);

/*
 * Pointer-table fold: the same chain over W independent arenas, without the
 * copy into a stacked buffer that the reference's `LoopbackWorld::run_round`
 * makes (mamba-rs src/dist/reducer.rs) -- the kernel reads every rank's
 * arena directly.
 *   out  device, len f32, written. It may be exactly one of the sources
 *        (out == srcs[k], the in-place fold of memra-engine 0.128.0
 *        tests/tp_ar_gpu.rs `memra_tp_ar_fold(dst, stage, ...)`); any other
 *        overlap with a source is DETFOLD_ERR_OVERLAP. Sources may overlap
 *        each other (they are only read).
 *   srcs host array of W device pointers, each to len f32, read.
 */
DETFOLD_API int detfold_sum_ptrs(float *out, const float *const *srcs, int W, int64_t len, void *stream);

/*
 * The mean as its own pass (mamba-rs src/dist/reducer.rs, module doc: the
 * caller multiplies the sum by 1/W): buf[i] = fl(buf[i] * scale), in place.
 *   buf device, len f32, read and written.
 * scale == 1.0f enqueues nothing.
 */
DETFOLD_API int detfold_scale(float *buf, int64_t len, float scale, void *stream);

/*
 * Fused loopback all-reduce, in place: for each i, read arenas[0..W-1][i],
 * fold in ascending rank order, multiply by mean_scale (skipped when it is
 * exactly 1.0f), and write the result to every arena. One pass replaces the
 * reference's exchange + fold + distribute (mamba-rs src/dist/reducer.rs,
 * `LoopbackWorld::run_round`, `reduce_sum_fixed_order_nccl`); the end state
 * is the same: every arena holds the identical ascending-rank sum.
 *   arenas host array of W device pointers, each to len f32, read and
 *          written. Arenas must be pairwise disjoint (DETFOLD_ERR_OVERLAP).
 * W == 1 leaves the arena as it is except for the mean multiply.
 */
DETFOLD_API int detfold_loopback_allreduce(float *const *arenas, int W, int64_t len, float mean_scale,
                               void *stream);

/*
 * The mean's scale (mamba-rs src/dist/reducer.rs, module doc: the sum is
 * multiplied by 1/W): *scale = fl(1/W), the binary32 reciprocal of W rounded
 * to nearest-even, exact for power-of-two W. Pass it as mean_scale.
 *   scale  host, written.
 * Host only; touches no device.
 */
DETFOLD_API int detfold_mean_scale(int W, float *scale);

/*
 * Library plumbing (the pages have no counterpart): bytes of device
 * workspace that the staged all-reduce needs for (len, W) -- W stack rows
 * of the largest owner shard, padded so that every row can share its source
 * shard's 32-byte phase. Returns a negative status for invalid len or W.
 */
DETFOLD_API int64_t detfold_staged_workspace_bytes(int64_t len, int W);

/*
 * Staged loopback all-reduce: the reference's own dataflow on one device
 * (mamba-rs src/dist/reducer.rs, `LoopbackWorld::run_round`), kept as the
 * comparator of the fused call. For each owner o with a non-empty shard
 * (detfold_shard_plan): copy every rank's slice of that shard into stack
 * slot = source rank, in ascending rank order, fold the slots into arena
 * o's shard, and apply mean_scale in the fold's store. Then copy every
 * owner's shard to all other arenas. The copies are pure byte movement: one
 * SM movement launch per phase and owner (the distribute phase reads the
 * owner's shard once for its W-1 destinations). Same end state and bits as
 * detfold_loopback_allreduce.
 *   arenas    host array of W device pointers (as above, pairwise disjoint).
 *   workspace device, >= detfold_staged_workspace_bytes(len, W) bytes,
 *             16-byte aligned, disjoint from every arena; contents on entry
 *             are ignored, on return undefined. Not needed when W == 1.
 * Unlike the reference, no stream synchronization happens between owners:
 * the workspace is caller-owned, so stream order alone protects its reuse.
 */
DETFOLD_API int detfold_loopback_allreduce_staged(float *const *arenas, int W, int64_t len,
                                      float mean_scale, void *workspace, int64_t workspace_bytes,
                                      void *stream);

/*
 * The staged all-reduce with the comparator's variants selected by `flags`
 * (DETFOLD_STAGED_* bits; flags == 0 is detfold_loopback_allreduce_staged):
 *   DETFOLD_STAGED_REVERSE_DELIVERY  copy the peers into the stack in
 *       descending rank order -- the slot, not the arrival order, fixes the
 *       chain, so the bits must not change (the page's delivery-order
 *       argument for `run_round`);
 *   DETFOLD_STAGED_SEPARATE_SCALE    the mean multiply as its own pass after
 *       each owner's fold, as the reference's caller applies it;
 *   DETFOLD_STAGED_CE_COPIES         move bytes with one cudaMemcpyAsync per
 *       copy (the copy engines), as the reference's `copy_d2d` does.
 * Any other bit is DETFOLD_ERR_ARG.
 */
DETFOLD_API int detfold_loopback_allreduce_staged_ex(float *const *arenas, int W, int64_t len,
                                         float mean_scale, int flags, void *workspace,
                                         int64_t workspace_bytes, void *stream);

/*
 * Pointer-table fold with the table in device memory. The kernel reads the
 * table when it runs, so a CUDA graph captured once follows new addresses
 * written into the table between replays (the rebind pattern of
 * memra-engine 0.136.0 tests/gdn_packed_gpu.rs, `packed_matches_per_row`
 * with graph_rebind). Same chain and bits as detfold_sum_ptrs.
 *   out       device, len f32, written; may be one of the sources.
 *   d_srcs    DEVICE array of W device pointers (8-byte aligned), read by the
 *             kernel; each entry must address len f32 that stay valid until
 *             the launch completes. Only the out == srcs[k] overlap is legal;
 *             the host cannot check this, so it is the caller's contract.
 *   d_status  optional DEVICE int (NULL = none): set to DETFOLD_OK, or to
 *             DETFOLD_ERR_NULL / DETFOLD_ERR_ALIGN when a table entry is NULL
 *             or not 4-byte aligned -- then nothing else is written. Not
 *             touched when the call returns before launching (len == 0 or
 *             a host-side error).
 */
DETFOLD_API int detfold_sum_ptrs_dev(float *out, const float *const *d_srcs, int W, int64_t len, int *d_status,
                         void *stream);

/*
 * Fused loopback all-reduce over a device-resident arena table (as
 * detfold_loopback_allreduce, with the table read by the kernel; arenas must
 * be pairwise disjoint -- the caller's contract). d_status as above.
 */
DETFOLD_API int detfold_loopback_allreduce_dev(float *const *d_arenas, int W, int64_t len, float mean_scale,
                                   int *d_status, void *stream);

/*
 * One-shot all-reduce, emulated on one device in a single cooperative launch
 * (memra-engine 0.128.0 tests/tp_ar_gpu.rs,
 * `one_shot_all_reduce_matches_the_host_sum_bitwise`). Each rank is a group of
 * CTAs. An entry barrier and an exit barrier made of per-CTA epoch flags
 * frame the fold: every rank folds all W arenas in ascending rank order into
 * its stage row, times mean_scale (skipped when exactly 1.0f), and after the
 * exit barrier copies the row into its own arena. End state and bits are
 * those of detfold_loopback_allreduce.
 *   arenas    host array of W <= DETFOLD_ONESHOT_MAX_W device pointers to len
 *             f32, pairwise disjoint.
 *   len       <= DETFOLD_ONESHOT_MAX_LEN (a small-payload primitive).
 *   link      device, DETFOLD_ONESHOT_LINK_BYTES, 8-byte aligned, zero-filled
 *             once before the first call on it, then reused unchanged: the
 *             entry and exit barrier flags and an epoch counter.
 *   epoch     0: the link's counter supplies the epoch (the largest epoch
 *             used on this link, plus one), so a call captured in a CUDA
 *             graph replays correctly. >= 1: this epoch, which must be larger
 *             than every epoch used before on this link. The barrier flags
 *             and the counter only grow, so nothing needs resetting after a
 *             refused call.
 *   stage     device, W * len f32 scratch, disjoint from the arenas.
 *   words     device, W ints: rank r's refusal word -- DETFOLD_OK, or
 *             DETFOLD_ONESHOT_REFUSE_ENTRY / _EXIT when its bounded wait at
 *             that barrier ran out, in which case its arena is untouched.
 *             Read the words before the numbers.
 *   wait_ns   bound on each barrier wait, 1 .. 2e9 ns (DETFOLD_ERR_ARG else).
 *   drop_rank -1, or a rank that leaves without publishing at one barrier
 *             (the entry barrier, or the exit barrier when drop_at_exit != 0)
 *             so that the others' waits run out: failure detection is tested
 *             this way, with no fault and no hang.
 * DETFOLD_ERR_CUDA with cudaErrorCooperativeLaunchTooLarge when W rank
 * groups cannot be co-resident.
 */
#define DETFOLD_ONESHOT_MAX_W 64
#define DETFOLD_ONESHOT_MAX_LEN ((int64_t)1 << 22)
#define DETFOLD_ONESHOT_MAX_CTAS 1024
#define DETFOLD_ONESHOT_LINK_BYTES (2 * DETFOLD_ONESHOT_MAX_CTAS * 8 + 64)
#define DETFOLD_ONESHOT_REFUSE_ENTRY 40043
#define DETFOLD_ONESHOT_REFUSE_EXIT 40044
DETFOLD_API int detfold_one_shot_allreduce(float *const *arenas, int W, int64_t len, float mean_scale,
                               void *link, uint64_t epoch, float *stage, int *words,
                               int64_t wait_ns, int drop_rank, int drop_at_exit, void *stream);

/*
 * Broadcast, pure byte movement (memra-engine 0.128.0 tests/tp_ar_gpu.rs,
 * `broadcast_and_all_gather_move_bytes_exactly`: rank 0's buffer lands on
 * every other rank byte for byte): dsts[k][i] = src[i] for every k.
 *   dsts  host array of ndst device pointers, each to len f32, written;
 *         pairwise disjoint and disjoint from src (DETFOLD_ERR_OVERLAP).
 *   src   device, len f32, read.
 * 1 <= ndst <= DETFOLD_MAX_W (DETFOLD_ERR_WORLD). One launch reads src once.
 */
DETFOLD_API int detfold_broadcast(float *const *dsts, int ndst, const float *src, int64_t len, void *stream);

/*
 * All-gather, pure byte movement (same test): every output receives the
 * concatenation of the W parts in rank order,
 *     outs[r][p * span + j] = parts[p][j]   for all r, p < W and j < span.
 *   outs   host array of W device pointers, each to W * span f32, written;
 *          pairwise disjoint and disjoint from every part.
 *   parts  host array of W device pointers, each to span f32, read (parts
 *          may overlap each other).
 * With W <= 8 and every pair at one 16-byte phase, one movement launch for
 * all pairs (each part read once); otherwise one launch per part.
 */
DETFOLD_API int detfold_all_gather(float *const *outs, int W, const float *const *parts, int64_t span,
                       void *stream);

/*
 * Contiguous owner shards (imported as `shard_plan` by mamba-rs
 * src/dist/reducer.rs; its body is not printed there). Reading: balanced,
 * shard r = {start = r*base + min(r, rem), len = base + (r < rem)} with
 * base = len / W, rem = len % W; shards may be empty when len < W.
 *   starts, lens  host arrays of W int64, written.
 * Host only; touches no device.
 */
DETFOLD_API int detfold_shard_plan(int64_t len, int W, int64_t *starts, int64_t *lens);

/*
 * Allocation-free staged loopback all-reduce. The sources have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- code
 * that runs while a stream is being captured into a CUDA graph (allocation
 * is not permitted there), and runtimes whose device memory is owned and
 * budgeted by their own allocator or reserved up front, where a stray
 * allocation would fail or break the budget. It computes exactly what
 * detfold_loopback_allreduce_staged_ex computes, with the same arguments
 * except the workspace: its scratch is a file-scope device array of
 * DETFOLD_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   - Requests whose workspace (detfold_staged_workspace_bytes(len, W)) is
 *     larger than DETFOLD_NOALLOC_SCRATCH_BYTES return
 *     DETFOLD_ERR_SCRATCH_LIMIT and enqueue nothing.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture.
 *   - Every call shares the one array. Calls that overlap on the GPU (on
 *     different streams without ordering between them) race on it; calls
 *     ordered on one stream are safe. Nothing in the array needs to start
 *     at zero: each call writes the stack rows before it reads them.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define DETFOLD_NOALLOC_SCRATCH_BYTES ((int64_t)16 << 20)
DETFOLD_API int detfold_loopback_allreduce_staged_noalloc(float *const *arenas, int W, int64_t len,
                                              float mean_scale, int flags, void *stream);

/* Library plumbing (no counterpart on the pages): a static, human-readable
 * name for a status code. */
DETFOLD_API const char *detfold_status_string(int status);

/*
 * Library plumbing (no counterpart on the pages): the cudaError_t value of
 * the last DETFOLD_ERR_CUDA returned on the calling thread (0 if none).
 */
DETFOLD_API int detfold_last_cuda_error(void);

/*
 * Library plumbing (no counterpart on the pages): number of bounded waits
 * that ran out, since the library was loaded, in the bulk-async (TMA)
 * pipelines that large aligned folds, all-reduces and moves use (W <= 8;
 * len >= 2^21 for folds over pointer tables passed from the host, len >= 2^20
 * for folds over device-resident tables and for moves). Each such wait
 * stops its CTA early, so any nonzero count
 * means some output is incomplete. It should always be 0; tests check that.
 * Synchronous: it reads a device counter (implicitly synchronizing the
 * device), so it is a diagnostic, not for hot loops.
 *   count  host, written.
 */
DETFOLD_API int detfold_pipeline_timeouts(int64_t *count);

#ifdef __cplusplus
}
#endif

#endif /* DETFOLD_H */
