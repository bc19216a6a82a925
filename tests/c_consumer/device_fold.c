/* A plain C consumer of libdetfold on the GPU, with the CUDA runtime's C API
 * for memory and no Python: reads W rows of n floats from argv[1], runs the
 * stacked fold and the fused all-reduce (mean scale argv[4]) on one stream,
 * and writes the fold, then every arena, to argv[2]. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "detfold.h"

#define CHECK(x)                                                                      \
    do {                                                                              \
        if ((x) != cudaSuccess) {                                                     \
            fprintf(stderr, "cuda error at line %d\n", __LINE__);                      \
            return 2;                                                                 \
        }                                                                             \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 5) return 1;
    const int W = atoi(argv[3]);
    const float scale = (float)atof(argv[4]);
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 1;
    fseek(f, 0, SEEK_END);
    const int64_t bytes = ftell(f);
    fseek(f, 0, SEEK_SET);
    const int64_t n = bytes / 4 / W;
    float *h = (float *)malloc((size_t)bytes);
    if (fread(h, 1, (size_t)bytes, f) != (size_t)bytes) return 1;
    fclose(f);

    float *d_stacked, *d_out, *d_arena[8];
    cudaStream_t st;
    CHECK(cudaStreamCreate(&st));
    CHECK(cudaMalloc((void **)&d_stacked, (size_t)bytes));
    CHECK(cudaMalloc((void **)&d_out, (size_t)n * 4));
    CHECK(cudaMemcpy(d_stacked, h, (size_t)bytes, cudaMemcpyHostToDevice));
    for (int r = 0; r < W; ++r) {
        CHECK(cudaMalloc((void **)&d_arena[r], (size_t)n * 4));
        CHECK(cudaMemcpy(d_arena[r], h + (int64_t)r * n, (size_t)n * 4, cudaMemcpyHostToDevice));
    }
    int rc = detfold_sum_stacked(d_out, d_stacked, W, n, st);
    if (rc) { fprintf(stderr, "sum_stacked: %s\n", detfold_status_string(rc)); return 3; }
    rc = detfold_loopback_allreduce(d_arena, W, n, scale, st);
    if (rc) { fprintf(stderr, "allreduce: %s\n", detfold_status_string(rc)); return 3; }
    CHECK(cudaStreamSynchronize(st));

    FILE *o = fopen(argv[2], "wb");
    float *tmp = (float *)malloc((size_t)n * 4);
    CHECK(cudaMemcpy(tmp, d_out, (size_t)n * 4, cudaMemcpyDeviceToHost));
    fwrite(tmp, 4, (size_t)n, o);
    for (int r = 0; r < W; ++r) {
        CHECK(cudaMemcpy(tmp, d_arena[r], (size_t)n * 4, cudaMemcpyDeviceToHost));
        fwrite(tmp, 4, (size_t)n, o);
    }
    fclose(o);
    printf("ok %lld\n", (long long)n);
    return 0;
}
