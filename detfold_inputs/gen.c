/*
 * Seeded synthetic input generators for the fixed-order fold.
 *
 * This module is shared by both sides of every parity check: the CPU oracle
 * and the CUDA path are each fed the arrays made here. It holds none of the
 * fold's arithmetic (no addition of rank addends, no mean scale); it only
 * turns seeds into f32 values.
 *
 * Every stream is the xorshift64 generator of memra-engine 0.128.0
 * tests/tp_ar_gpu.rs (`vecf`): state = seed * 0x9E3779B97F4A7C15 | 1, then
 * per draw x ^= x << 13; x ^= x >> 7; x ^= x << 17. `vecf` maps the top 24
 * bits to [-1, 1); continuous draws use the top 53 bits as in `varied` of
 * memra-engine 0.136.0 tests/gdn_packed_gpu.rs.
 *
 * Kinds (one row of `n` values per seed):
 *   0 VECF      ((x >> 40) / 2^24 - 0.5) * 2, all arithmetic in f32 (exact).
 *   1 GRADIENT  v = f32(1e-3 * z), z ~ N(0,1) by Box-Muller from two 53-bit
 *               draws; with a third draw < 0.01, v = f32(v * 1000).
 *   2 NORMAL    f32(z), z ~ N(0,1) by Box-Muller.
 *   3 STRESS    signed zero with p = 0.01, else a random nonzero subnormal
 *               with p = 0.001, else magnitude 10^(-30 + 34u) rounded to f32;
 *               random sign. Elements 0..15 of each row are then overwritten
 *               by fixed special columns (see stress_specials).
 *
 * Rows are independent streams, so multi-row fills run one thread per row.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { KIND_VECF = 0, KIND_GRADIENT = 1, KIND_NORMAL = 2, KIND_STRESS = 3 };

static inline uint64_t xs_init(uint64_t seed) { return seed * 0x9E3779B97F4A7C15ULL | 1ULL; }

static inline uint64_t xs_next(uint64_t *s)
{
    uint64_t x = *s;
    x ^= x << 13;
    x ^= x >> 7;
    x ^= x << 17;
    *s = x;
    return x;
}

/* [0, 1) from the top 53 bits. */
static inline double u53(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

static inline float f32_from_bits(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static double box_muller(uint64_t *s)
{
    double u1 = 1.0 - u53(xs_next(s)); /* (0, 1]: log stays finite */
    double u2 = u53(xs_next(s));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/*
 * Fixed special columns for the stress rows, chosen so that the fold's
 * sign-of-zero, subnormal, cancellation and order rules all show up in the
 * first 16 elements. Rank r of W writes its own entry of each column.
 */
static void stress_specials(float *row, int64_t n, int r, int W)
{
    float v[16];
    v[0] = -0.0f;                                   /* all -0            */
    v[1] = 0.0f;                                    /* all +0            */
    v[2] = (r == 0) ? -0.0f : 0.0f;                 /* -0 then +0s       */
    v[3] = (r == W - 1) ? 0.0f : -0.0f;             /* -0s then +0       */
    v[4] = (r == 0) ? 1536.0f : (r == 1) ? -1536.0f : 0.0f;        /* x, -x  */
    v[5] = (r == 0) ? f32_from_bits(0x0020B6A3u)                    /* subnormal pair */
         : (r == 1) ? f32_from_bits(0x8020B6A3u) : -0.0f;
    v[6] = f32_from_bits(0x00000001u);              /* all 2^-149        */
    v[7] = 1.0f;                                    /* all ones          */
    v[8] = (r == 0) ? 16777216.0f : 1.0f;           /* 2^24 then ones    */
    v[9] = (r == W - 1) ? 16777216.0f : 1.0f;       /* ones then 2^24    */
    v[10] = (r == 0) ? 1.0e8f : (r == 1) ? 1.0f : (r == 2) ? -1.0e8f : 0.5f;
    v[11] = (r & 1) ? -3.0e-38f : 3.0e-38f;          /* normal/subnormal edge */
    v[12] = f32_from_bits(0x007FFFFFu);             /* all max subnormal */
    v[13] = (r == 0) ? 1.0f : f32_from_bits(0x33800000u); /* 1 then 2^-24s */
    v[14] = (r == 0) ? f32_from_bits(0x33800000u) : (r == 1) ? f32_from_bits(0x33800000u) : 1.0f;
    v[15] = (r % 3 == 0) ? 1.0e4f : (r % 3 == 1) ? -9999.5f : 2.5e-4f;
    for (int i = 0; i < 16 && i < n; ++i) row[i] = v[i];
}

static void fill_row(int kind, float *out, int64_t n, uint64_t seed, int r, int W)
{
    uint64_t s = xs_init(seed);
    switch (kind) {
    case KIND_VECF:
        for (int64_t i = 0; i < n; ++i) {
            uint64_t x = xs_next(&s);
            out[i] = ((float)(x >> 40) / 16777216.0f - 0.5f) * 2.0f;
        }
        break;
    case KIND_GRADIENT:
        for (int64_t i = 0; i < n; ++i) {
            double z = box_muller(&s);
            double u3 = u53(xs_next(&s));
            float v = (float)(1.0e-3 * z);
            if (u3 < 0.01) v = v * 1000.0f;
            out[i] = v;
        }
        break;
    case KIND_NORMAL:
        for (int64_t i = 0; i < n; ++i) out[i] = (float)box_muller(&s);
        break;
    case KIND_STRESS:
        for (int64_t i = 0; i < n; ++i) {
            double u = u53(xs_next(&s));
            uint64_t bits = xs_next(&s);
            uint32_t sign = (uint32_t)(bits >> 63) << 31;
            float v;
            if (u < 0.01) {
                v = f32_from_bits(sign);
            } else if (u < 0.011) {
                uint32_t m = (uint32_t)(bits >> 20) & 0x7FFFFFu;
                if (m == 0) m = 1;
                v = f32_from_bits(sign | m);
            } else {
                float mag = (float)pow(10.0, -30.0 + 34.0 * u53(xs_next(&s)));
                v = sign ? -mag : mag;
            }
            out[i] = v;
        }
        stress_specials(out, n, r, W);
        break;
    default:
        break;
    }
}

struct rows_job {
    int kind;
    float *base;
    int64_t n, row_stride;
    uint64_t seed0, seed_step;
    int W, r_begin, r_step;
};

static void *rows_worker(void *p)
{
    struct rows_job *j = (struct rows_job *)p;
    for (int r = j->r_begin; r < j->W; r += j->r_step)
        fill_row(j->kind, j->base + (int64_t)r * j->row_stride, j->n,
                 j->seed0 + j->seed_step * (uint64_t)r, r, j->W);
    return NULL;
}

/*
 * Fill W rows of n values; row r starts at out + r * row_stride and uses seed
 * seed0 + seed_step * r. Up to `threads` threads, one row at a time each.
 * Returns 0, or -1 on a bad argument.
 */
int detfold_gen_rows(int kind, float *out, int64_t W, int64_t n, int64_t row_stride,
                     uint64_t seed0, uint64_t seed_step, int threads)
{
    if (!out || W < 1 || W > 4096 || n < 0 || row_stride < n || kind < 0 || kind > 3) return -1;
    if (threads < 1) threads = 1;
    if (threads > W) threads = (int)W;
    if (threads > 64) threads = 64;
    struct rows_job jobs[64];
    pthread_t tid[64];
    int started[64] = {0};
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (struct rows_job){kind, out, n, row_stride, seed0, seed_step, (int)W, t, threads};
        if (t > 0) started[t] = pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) == 0;
    }
    rows_worker(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (started[t]) {
            pthread_join(tid[t], NULL);
        } else {
            rows_worker(&jobs[t]); /* thread creation failed: do it here */
        }
    }
    return 0;
}
