/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, serial, single-threaded CPU statement of what the fixed-order fold
 * computes. Only the test suite, the smoke check and the benchmark's CPU
 * baseline may load it. It shares no code with the CUDA library: no headers,
 * no helpers, no tables.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, no
 * flush-to-zero, IEEE binary32 round-to-nearest-even on x86-64 and aarch64).
 *
 * Sources (docs.rs pages):
 *   [reducer]  mamba-rs 0.6.2 src/dist/reducer.rs
 *                - module doc: ascending source-rank fold, sum then a separate
 *                  multiply by 1/W for the mean;
 *                - `reduce_sum_reference`: acc = addends[0][i]; acc += a[i] for
 *                  the remaining addends in order;
 *                - `LoopbackWorld::run_round`: per-owner exchange into slots
 *                  indexed by source rank, fold, then distribute.
 *   [tp_ar]    memra-engine 0.128.0 tests/tp_ar_gpu.rs (bitwise host sum).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - IEEE binary32, round-to-nearest-even, subnormals kept (no FTZ).
 *   - The mean is fl(sum * fl(1/W)), one rounded multiply, not a division.
 *     A mean_scale of exactly 1.0f means "no multiply".
 *   - shard_plan is not printed on the pages: balanced contiguous shards,
 *     the first len % W owners one element longer.
 *
 * Parity pins: every function here is pinned by tests that do not call it to
 * compute their expectation (exact rational IEEE model, closed forms,
 * brute-force rank orders, invariants); see tests/test_oracle_pins.py.
 */
#include <stdint.h>
#include <string.h>

/* [reducer] `reduce_sum_reference`: per element, the W addends in ascending
 * source-rank order, starting from addend 0 (not from 0.0). */
void oracle_fold(const float *const *srcs, int W, int64_t len, float *out)
{
    for (int64_t i = 0; i < len; ++i) {
        float acc = srcs[0][i];
        for (int r = 1; r < W; ++r) acc = acc + srcs[r][i];
        out[i] = acc;
    }
}

/* [reducer] `DET_SUM_RANKS_SRC` layout: stacked is [W][len], slot = source rank. */
void oracle_fold_stacked(const float *stacked, int W, int64_t len, float *out)
{
    for (int64_t i = 0; i < len; ++i) {
        float acc = stacked[i];
        for (int r = 1; r < W; ++r) acc = acc + stacked[(int64_t)r * len + i];
        out[i] = acc;
    }
}

/* [reducer] module doc: the mean multiplies the sum by 1/W (here fl(1/W)). */
float oracle_mean_scale(int W)
{
    return 1.0f / (float)W;
}

/* [reducer] module doc: the separate mean multiply. */
void oracle_scale(float *buf, int64_t len, float scale)
{
    if (scale == 1.0f) return;
    for (int64_t i = 0; i < len; ++i) buf[i] = buf[i] * scale;
}

/*
 * The all-reduce's end state: every arena holds the fold of all arenas' old
 * values, times scale. (W arenas of len f32, pairwise disjoint.)
 * [reducer] module doc + `LoopbackWorld::run_round` ("every arena holds the
 * identical ascending-rank sum").
 */
void oracle_allreduce(float *const *arenas, int W, int64_t len, float scale)
{
    for (int64_t i = 0; i < len; ++i) {
        float acc = arenas[0][i];
        for (int r = 1; r < W; ++r) acc = acc + arenas[r][i];
        if (scale != 1.0f) acc = acc * scale;
        for (int r = 0; r < W; ++r) arenas[r][i] = acc;
    }
}

/* Balanced contiguous owner shards (reading: the pages import shard_plan
 * without printing it). Shard r = {r*base + min(r, rem), base + (r < rem)}. */
void oracle_shard_plan(int64_t len, int W, int64_t *starts, int64_t *lens)
{
    int64_t base = len / W, rem = len % W;
    for (int r = 0; r < W; ++r) {
        starts[r] = (int64_t)r * base + (r < rem ? r : rem);
        lens[r] = base + (r < rem ? 1 : 0);
    }
}

/*
 * [reducer] `LoopbackWorld::run_round`, the reference's dataflow on the host:
 * phase A, per owner with a non-empty shard, copies every rank's slice of
 * that shard into stack slot = source rank (ascending, or descending when
 * `reverse` is set -- the result must not change), folds the slots in
 * ascending slot order into the owner's shard, and (reading) applies the
 * mean multiply there; phase B copies each owner's shard to every other
 * arena. `stack` holds at least W * max shard length floats.
 */
void oracle_staged_allreduce(float *const *arenas, int W, int64_t len, float scale,
                             int reverse, float *stack)
{
    int64_t starts[W], lens[W];
    oracle_shard_plan(len, W, starts, lens);
    for (int o = 0; o < W; ++o) {
        int64_t s = starts[o], n = lens[o];
        if (n == 0) continue;
        for (int k = 0; k < W; ++k) {
            int src = reverse ? W - 1 - k : k;
            memcpy(stack + (int64_t)src * n, arenas[src] + s, (size_t)n * sizeof(float));
        }
        oracle_fold_stacked(stack, W, n, arenas[o] + s);
        oracle_scale(arenas[o] + s, n, scale);
    }
    for (int o = 0; o < W; ++o) {
        if (lens[o] == 0) continue;
        for (int r = 0; r < W; ++r) {
            if (r == o) continue;
            memcpy(arenas[r] + starts[o], arenas[o] + starts[o], (size_t)lens[o] * sizeof(float));
        }
    }
}

/* memra-engine 0.136.0 tests/gdn_packed_gpu.rs `bit_diffs`: words whose bit
 * patterns differ. */
int64_t oracle_bit_diffs(const float *a, const float *b, int64_t n)
{
    int64_t d = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t x, y;
        memcpy(&x, a + i, 4);
        memcpy(&y, b + i, 4);
        d += (x != y);
    }
    return d;
}
