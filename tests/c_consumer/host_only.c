/* A plain C consumer of libdetfold's host-only entry points (no GPU needed):
 * shard plan, status strings, workspace sizing and argument validation. */
#include <stdint.h>
#include <stdio.h>

#include "detfold.h"

int main(void)
{
    int64_t starts[6], lens[6];
    if (detfold_shard_plan((1 << 20) + 7, 6, starts, lens) != DETFOLD_OK) return 1;
    for (int r = 0; r < 6; ++r) printf("shard %d %lld %lld\n", r, (long long)starts[r], (long long)lens[r]);
    printf("ws %lld\n", (long long)detfold_staged_workspace_bytes(100000000, 4));
    printf("null %d\n", detfold_sum_stacked(0, 0, 2, 8, 0));
    printf("world %d\n", detfold_sum_ptrs((float *)64, (const float *const *)64, 0, 8, 0));
    printf("zero %d\n", detfold_scale((float *)64, 0, 0.5f, 0));
    printf("str %s\n", detfold_status_string(DETFOLD_ERR_OVERLAP));
    return 0;
}
