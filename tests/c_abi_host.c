/* A plain C99 caller of libgb's host-only entry points: it builds against
 * include/gb.h alone, links libgb.so, and needs no GPU.  Prints one line per
 * check as "name value" for the test that compiles and runs it. */
#include <stdio.h>
#include <string.h>

#include "gb.h"

int main(void)
{
    gb_ctx *ctx = NULL;
    const int sizes[3] = {2, 3, 1};
    gb_status st = gb_create(&ctx, 3, sizes);
    printf("create %d\n", (int)st);
    if (st != GB_OK)
        return 1;
    printf("world %d\n", gb_world_size(ctx));
    printf("islands %d\n", gb_n_islands(ctx));
    printf("first2 %d\n", gb_island_first_rank(ctx, 2));
    printf("island_of4 %d\n", gb_island_of_rank(ctx, 4));
    printf("payload_e4m3 %zu\n", gb_payload_bytes(GB_CODEC_E4M3, 256, (size_t)6553600));
    printf("payload_bf16 %zu\n", gb_payload_bytes(GB_CODEC_BF16, 256, (size_t)1000));
    printf("scales_off %zu\n", gb_payload_scales_offset(GB_CODEC_E5M2, 128, (size_t)1001));

    /* an argument error answers before any CUDA call and is not sticky */
    void *bufs[6] = {0};
    st = gb_all_reduce(ctx, bufs, 10, GB_F32, GB_SUM, GB_CODEC_NONE, 256, NULL);
    printf("null_bufs %d\n", (int)st);
    printf("sticky %d\n", (int)gb_context_status(ctx));
    printf("status_string %s\n", gb_status_string(GB_ERR_MISALIGNED));

    /* bucket plan: 5 tensors of float32 under a 4000-byte cap */
    const size_t numel[5] = {600, 500, 1200, 10, 990};
    int bucket_of[5];
    size_t offset[5], bucket_numel[5];
    int nb = 0;
    st = gb_bucket_plan(numel, 5, 4, 4000, 1, bucket_of, offset, bucket_numel, 5, &nb);
    printf("plan %d %d", (int)st, nb);
    for (int b = 0; b < nb; ++b)
        printf(" %zu", bucket_numel[b]);
    printf("\n");
    printf("destroy %d\n", (int)gb_destroy(ctx));
    return 0;
}
