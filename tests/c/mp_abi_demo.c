/*
 * A C caller of libmp.so: only include/mp.h and the CUDA runtime, no Python.
 *
 * 1. The worked example of make_row_id_map ("d9d 0.1.0 -- d9d/kernel/moe/
 *    permute_with_probs.py"): 5 tokens, 3 experts, routing map
 *    [[1,1,0],[1,0,1],[0,0,1],[1,1,0],[0,0,0]], written as top-2 expert ids
 *    with -1 for an empty slot.  The page's pass-2 destinations give
 *    row_id_map [[0,3],[1,5],[6,-1],[2,4],[-1,-1]] and offsets [0,3,5,7].
 * 2. permute then unpermute with unit probabilities: token t comes back
 *    multiplied by its number of routed slots (small integers: exact).
 * 3. A host-detected error: H = 0 gives MP_ERR_INVALID_ARG, nothing launched.
 * Prints "ok" and returns 0 when everything matches.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mp.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            return 1;                                                              \
        }                                                                          \
    } while (0)

#define CHECK_MP(x)                                                                \
    do {                                                                           \
        mp_status_t s_ = (x);                                                      \
        if (s_ != MP_OK) {                                                         \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, mp_status_string(s_)); \
            return 1;                                                              \
        }                                                                          \
    } while (0)

enum { T = 5, K = 2, E = 3, H = 16 };

/* bf16 bits of a small integer (exact: 8 significant bits suffice) */
static uint16_t bf16_of_int(int v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

int main(void)
{
    const int32_t idx[T * K] = {0, 1, 0, 2, 2, -1, 0, 1, -1, -1};
    const int32_t want_map[T * K] = {0, 3, 1, 5, 6, -1, 2, 4, -1, -1};
    const int32_t want_off[E + 1] = {0, 3, 5, 7};
    const int routed_slots[T] = {2, 2, 1, 2, 0};

    int32_t *d_idx, *d_map, *d_s2f, *d_counts, *d_off;
    void *d_ws;
    size_t ws_bytes = mp_build_map_workspace_size(T, K, E);
    if (ws_bytes == 0) return 1;
    CHECK_CUDA(cudaMalloc((void **)&d_idx, sizeof idx));
    CHECK_CUDA(cudaMalloc((void **)&d_map, sizeof idx));
    CHECK_CUDA(cudaMalloc((void **)&d_s2f, sizeof idx));
    CHECK_CUDA(cudaMalloc((void **)&d_counts, E * sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc((void **)&d_off, (E + 1) * sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(d_idx, idx, sizeof idx, cudaMemcpyHostToDevice));

    /* 1. the worked example */
    CHECK_MP(mp_build_map(d_idx, T, K, E, d_map, d_s2f, d_counts, d_off, d_ws, ws_bytes, NULL,
                          NULL));
    int32_t map[T * K], off[E + 1];
    CHECK_CUDA(cudaMemcpy(map, d_map, sizeof map, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(off, d_off, sizeof off, cudaMemcpyDeviceToHost));
    if (memcmp(map, want_map, sizeof map) || memcmp(off, want_off, sizeof off)) {
        fprintf(stderr, "row_id_map or offsets differ from the worked example\n");
        return 1;
    }

    /* 2. permute, then unpermute with unit probabilities */
    uint16_t x[T * H], y[T * H];
    float probs[T * K];
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) x[t * H + h] = bf16_of_int(t * H + h - 40);
    for (int i = 0; i < T * K; ++i) probs[i] = 1.0f;
    mp_bf16_t *d_x, *d_rows, *d_y;
    float *d_probs, *d_rows_p;
    CHECK_CUDA(cudaMalloc((void **)&d_x, sizeof x));
    CHECK_CUDA(cudaMalloc((void **)&d_y, sizeof y));
    CHECK_CUDA(cudaMalloc((void **)&d_rows, (size_t)T * K * H * sizeof(uint16_t)));
    CHECK_CUDA(cudaMalloc((void **)&d_probs, sizeof probs));
    CHECK_CUDA(cudaMalloc((void **)&d_rows_p, sizeof probs));
    CHECK_CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_probs, probs, sizeof probs, cudaMemcpyHostToDevice));
    CHECK_MP(mp_permute(d_x, d_probs, d_map, T, K, H, d_rows, d_rows_p, NULL));
    CHECK_MP(mp_unpermute(d_rows, d_probs, d_map, T, K, H, d_y, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_CUDA(cudaMemcpy(y, d_y, sizeof y, cudaMemcpyDeviceToHost));
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            const uint16_t want = bf16_of_int(routed_slots[t] * (t * H + h - 40));
            if (y[t * H + h] != want) {
                fprintf(stderr, "y[%d,%d] = 0x%04x, want 0x%04x\n", t, h, y[t * H + h], want);
                return 1;
            }
        }

    /* 3. a host-detected error: nothing is launched */
    if (mp_permute(d_x, NULL, d_map, T, K, 0, d_rows, NULL, NULL) != MP_ERR_INVALID_ARG) {
        fprintf(stderr, "H = 0 was not rejected\n");
        return 1;
    }

    cudaFree(d_idx);
    cudaFree(d_map);
    cudaFree(d_s2f);
    cudaFree(d_counts);
    cudaFree(d_off);
    cudaFree(d_ws);
    cudaFree(d_x);
    cudaFree(d_y);
    cudaFree(d_rows);
    cudaFree(d_probs);
    cudaFree(d_rows_p);
    printf("ok\n");
    return 0;
}
