/* A plain C99 caller of libgb on the GPU: it builds against include/gb.h and
 * the CUDA runtime's C API alone, all_reduces four rank buffers (2 islands
 * of 2, AVG, E4M3 with a scale per 256 elements) and reduce_scatters them,
 * and writes the results' raw bytes to the file named by argv[1]:
 * 4 x n float32 (all_reduce, ranks in order), then 4 x n/4 float32
 * (reduce_scatter slices).  The inputs are exact small binary fractions
 * from a fixed formula, so the test can rebuild them.  Exit status 0 on
 * success. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "gb.h"

#define N 70003u /* not a multiple of 256: a ragged last tile */
#define NRS 70004u /* a multiple of 4 for reduce_scatter */

static float value(unsigned r, unsigned j, unsigned salt)
{
    return (float)((int)((j * 7u + r * 13u + salt) % 101u) - 50) * 0.25f;
}

static int check(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

int main(int argc, char **argv)
{
    if (argc != 2)
        return 2;
    FILE *out = fopen(argv[1], "wb");
    if (!out)
        return 2;
    const int sizes[2] = {2, 2};
    gb_ctx *ctx = NULL;
    if (gb_create(&ctx, 2, sizes) != GB_OK)
        return 3;
    float *host = (float *)malloc(sizeof(float) * NRS);
    void *bufs[4] = {0}, *slices[4] = {0};
    for (unsigned r = 0; r < 4; ++r) {
        if (check(cudaMalloc(&bufs[r], sizeof(float) * NRS), "cudaMalloc") ||
            check(cudaMalloc(&slices[r], sizeof(float) * (NRS / 4)), "cudaMalloc"))
            return 4;
        for (unsigned j = 0; j < N; ++j)
            host[j] = value(r, j, 0);
        if (check(cudaMemcpy(bufs[r], host, sizeof(float) * N, cudaMemcpyHostToDevice), "to device"))
            return 4;
    }
    gb_status st = gb_all_reduce(ctx, bufs, N, GB_F32, GB_AVG, GB_CODEC_E4M3, 256, NULL);
    if (st != GB_OK) {
        fprintf(stderr, "gb_all_reduce: %s (%s)\n", gb_status_string(st), gb_last_error_message(ctx));
        return 5;
    }
    if (check(cudaDeviceSynchronize(), "synchronize"))
        return 5;
    for (unsigned r = 0; r < 4; ++r) {
        if (check(cudaMemcpy(host, bufs[r], sizeof(float) * N, cudaMemcpyDeviceToHost), "to host"))
            return 6;
        fwrite(host, sizeof(float), N, out);
    }
    /* reduce_scatter of fresh inputs, SUM, bf16 codec */
    for (unsigned r = 0; r < 4; ++r) {
        for (unsigned j = 0; j < NRS; ++j)
            host[j] = value(r, j, 5);
        if (check(cudaMemcpy(bufs[r], host, sizeof(float) * NRS, cudaMemcpyHostToDevice), "to device"))
            return 7;
    }
    st = gb_reduce_scatter(ctx, (const void *const *)bufs, slices, NRS, GB_F32, GB_SUM, GB_CODEC_BF16, 256, NULL);
    if (st != GB_OK) {
        fprintf(stderr, "gb_reduce_scatter: %s (%s)\n", gb_status_string(st), gb_last_error_message(ctx));
        return 8;
    }
    if (check(cudaDeviceSynchronize(), "synchronize"))
        return 8;
    for (unsigned r = 0; r < 4; ++r) {
        if (check(cudaMemcpy(host, slices[r], sizeof(float) * (NRS / 4), cudaMemcpyDeviceToHost), "to host"))
            return 9;
        fwrite(host, sizeof(float), NRS / 4, out);
    }
    fclose(out);
    for (unsigned r = 0; r < 4; ++r) {
        cudaFree(bufs[r]);
        cudaFree(slices[r]);
    }
    free(host);
    return gb_destroy(ctx) == GB_OK ? 0 : 10;
}
