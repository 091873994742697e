/*
 * A plain C caller of libasyncpipe: device memory from cudaMalloc, no Python,
 * no torch. Checks that the C interface is usable on its own: a pipelined
 * scale, the 64 x 4 row shift of the TIRx worked example, a cluster hand-off,
 * argument errors and status strings. Exit status 0 when every check passes.
 * With --no-gpu it only exercises the argument checks (no CUDA call is made).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "asyncpipe.h"
#include "asyncpipe_debug.h"

static int failures = 0;

#define CHECK(cond, ...)                         \
    do {                                         \
        if (!(cond)) {                           \
            fprintf(stderr, "FAIL: " __VA_ARGS__); \
            fprintf(stderr, "\n");               \
            ++failures;                          \
        }                                        \
    } while (0)

static void argument_checks(void) {
    float* fake = (float*)(uintptr_t)0x7f0000000000ull;
    CHECK(ap_scale(fake, fake + 4096, 4, 256, 2.0f, 1, 0) == AP_ERR_STAGES, "stages 1 accepted");
    CHECK(ap_scale(NULL, fake, 4, 256, 2.0f, 2, 0) == AP_ERR_NULL, "null input accepted");
    CHECK(ap_row_roll(fake, fake, 64, 4, 1, 0) == AP_ERR_ALIAS, "in-place roll accepted");
    CHECK(ap_cluster_exchange(fake, fake + (1 << 20), 1 << 20, 3, 32768, 0) == AP_ERR_CLUSTER, "cluster 3 accepted");
    CHECK(ap_scale(NULL, NULL, 0, 256, 2.0f, 2, 0) == AP_OK, "empty call not a no-op");
    CHECK(strcmp(ap_status_string(AP_ERR_ALIGN), "AP_ERR_ALIGN") == 0, "status string");
    CHECK(ap_debug_get(AP_DBG_TIMEOUT_NS) > 0, "default wait limit");
}

static int gpu_checks(void) {
    const int64_t n_tiles = 4099, tile = 256, n = n_tiles * tile;
    float* h_in = (float*)malloc((size_t)n * sizeof(float));
    float* h_out = (float*)malloc((size_t)n * sizeof(float));
    float *d_in = NULL, *d_out = NULL;
    if (!h_in || !h_out) return 1;
    for (int64_t i = 0; i < n; ++i) h_in[i] = (float)(i % 4093) * 0.25f - 511.0f;  /* exact in fp32 */
    if (cudaMalloc((void**)&d_in, (size_t)n * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&d_out, (size_t)n * sizeof(float)) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    cudaMemcpy(d_in, h_in, (size_t)n * sizeof(float), cudaMemcpyHostToDevice);

    /* pipelined scale: doubling is exact */
    CHECK(ap_scale(d_in, d_out, n_tiles, tile, 2.0f, 2, 0) == AP_OK, "ap_scale launch");
    CHECK(ap_check(0) == AP_OK, "ap_scale status");
    cudaMemcpy(h_out, d_out, (size_t)n * sizeof(float), cudaMemcpyDeviceToHost);
    for (int64_t i = 0; i < n; ++i) {
        if (h_out[i] != h_in[i] + h_in[i]) {
            CHECK(0, "ap_scale element %lld", (long long)i);
            break;
        }
    }

    /* the 64 x 4 row shift: B[i][j] = A[(i + 1) % 64][j] */
    CHECK(ap_row_roll(d_in, d_out, 64, 4, 1, 0) == AP_OK, "ap_row_roll launch");
    CHECK(ap_check(0) == AP_OK, "ap_row_roll status");
    cudaMemcpy(h_out, d_out, 256 * sizeof(float), cudaMemcpyDeviceToHost);
    for (int i = 0; i < 64; ++i)
        for (int j = 0; j < 4; ++j)
            if (h_out[i * 4 + j] != h_in[((i + 1) % 64) * 4 + j]) CHECK(0, "roll row %d col %d", i, j);

    /* cluster hand-off, clusters of 4, 16 KiB chunks: out chunk r = in chunk (r + 1) mod 4 */
    const int64_t chunk = 4096, groups = 8, m = groups * 4 * chunk;
    CHECK(ap_cluster_exchange(d_in, d_out, m, 4, chunk * 4, 0) == AP_OK, "exchange launch");
    CHECK(ap_check(0) == AP_OK, "exchange status");
    cudaMemcpy(h_out, d_out, (size_t)m * sizeof(float), cudaMemcpyDeviceToHost);
    for (int64_t c = 0; c < groups * 4; ++c) {
        const int64_t src = (c / 4) * 4 + (c % 4 + 1) % 4;
        if (memcmp(h_out + c * chunk, h_in + src * chunk, (size_t)chunk * sizeof(float)) != 0)
            CHECK(0, "exchange chunk %lld", (long long)c);
    }
    cudaFree(d_in);
    cudaFree(d_out);
    free(h_in);
    free(h_out);
    return 0;
}

int main(int argc, char** argv) {
    argument_checks();
    if (!(argc > 1 && strcmp(argv[1], "--no-gpu") == 0)) {
        if (gpu_checks() != 0) ++failures;
    }
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("c abi ok\n");
    return 0;
}
