/*
 * A plain C consumer of the library: only include/moe_route.h and the CUDA
 * runtime API, no Python and no torch.  One small layer (4 ranks, 16 experts,
 * top-2, H = 256, one empty rank) goes route -> dispatch -> identity expert
 * stand-in -> combine, and the program checks what the definitions fix:
 *   - the counts add up to T*K, and each rank's counts to B[s]*K;
 *   - tok2row and row2src are inverse maps of [0, T*K);
 *   - every dispatched row is its source token, bit for bit;
 *   - with identity experts and weights that sum to one, combine returns each
 *     token within one bf16 rounding.
 * Exit status 0 on success; it prints what failed otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_route.h"

enum { R = 4, E = 16, K = 2, H = 256 };

static float bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t lcg(uint32_t *s)
{
    *s = *s * 1664525u + 1013904223u;
    return *s >> 8;
}

#define CK(x)                                                                           \
    do {                                                                                \
        cudaError_t e_ = (x);                                                           \
        if (e_ != cudaSuccess) {                                                        \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                    \
            return 2;                                                                   \
        }                                                                               \
    } while (0)
#define MK(x)                                                                           \
    do {                                                                                \
        int s_ = (x);                                                                   \
        if (s_ != MOE_OK) {                                                             \
            fprintf(stderr, "%s: %s\n", #x, moe_strerror(s_));                          \
            return 3;                                                                   \
        }                                                                               \
    } while (0)
#define REQUIRE(c, ...)                                                                 \
    do {                                                                                \
        if (!(c)) {                                                                     \
            fprintf(stderr, __VA_ARGS__);                                               \
            fprintf(stderr, "\n");                                                      \
            return 1;                                                                   \
        }                                                                               \
    } while (0)

int main(void)
{
    const int32_t B[R] = {7, 0, 19, 6};
    int T = 0;
    for (int s = 0; s < R; ++s) T += B[s];
    const int rows = T * K;

    /* host inputs: x as bf16 bit patterns of moderate values, logits in [-2, 2) */
    uint16_t *x = malloc(sizeof(uint16_t) * (size_t)T * H);
    float *lg = malloc(sizeof(float) * (size_t)T * E);
    uint32_t st = 12345u;
    for (int i = 0; i < T * H; ++i) {
        uint32_t m = lcg(&st);
        x[i] = (uint16_t)(((m & 1u) << 15) | ((120u + (m >> 1) % 16u) << 7) | ((m >> 5) & 0x7fu));
    }
    for (int i = 0; i < T * E; ++i) lg[i] = (float)(lcg(&st) % 4096u) / 1024.0f - 2.0f;

    void *d_x, *d_lg, *d_idx, *d_w, *d_recv, *d_counts, *d_off, *d_eo, *d_t2r, *d_r2s, *d_y, *d_out, *d_ws;
    const size_t wsb = moe_dispatch_workspace_bytes(R, E, K, T);
    REQUIRE(wsb > 0, "workspace size 0");
    CK(cudaMalloc(&d_x, sizeof(uint16_t) * (size_t)T * H));
    CK(cudaMalloc(&d_lg, sizeof(float) * (size_t)T * E));
    CK(cudaMalloc(&d_idx, sizeof(int32_t) * (size_t)rows));
    CK(cudaMalloc(&d_w, sizeof(float) * (size_t)rows));
    CK(cudaMalloc(&d_recv, sizeof(uint16_t) * (size_t)rows * H));
    CK(cudaMalloc(&d_counts, sizeof(int32_t) * E * R));
    CK(cudaMalloc(&d_off, sizeof(int32_t) * (E * R + 1)));
    CK(cudaMalloc(&d_eo, sizeof(int32_t) * (E + 1)));
    CK(cudaMalloc(&d_t2r, sizeof(int32_t) * (size_t)rows));
    CK(cudaMalloc(&d_r2s, sizeof(int32_t) * (size_t)rows));
    CK(cudaMalloc(&d_y, sizeof(uint16_t) * (size_t)rows * H));
    CK(cudaMalloc(&d_out, sizeof(uint16_t) * (size_t)T * H));
    CK(cudaMalloc(&d_ws, wsb));
    CK(cudaMemcpy(d_x, x, sizeof(uint16_t) * (size_t)T * H, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_lg, lg, sizeof(float) * (size_t)T * E, cudaMemcpyHostToDevice));

    MK(moe_route_topk(d_lg, T, E, K, d_idx, d_w, 0));
    MK(moe_dispatch(d_x, d_idx, R, B, E, K, H, MOE_DTYPE_BF16, d_recv, NULL, d_counts, d_off, d_eo, d_t2r, d_r2s,
                    d_ws, wsb, 0));
    MK(moe_expert_scale(d_recv, NULL, MOE_DTYPE_BF16, d_eo, E, H, rows, 1, d_y, 0));
    MK(moe_combine(d_y, d_t2r, d_w, T, K, H, MOE_DTYPE_BF16, d_out, 0));
    int32_t code = -1;
    MK(moe_get_device_error(d_ws, &code, 0));   /* synchronises the stream */
    REQUIRE(code == 0, "device error word %#x", (unsigned)code);

    int32_t *counts = malloc(sizeof(int32_t) * E * R), *t2r = malloc(sizeof(int32_t) * rows);
    int32_t *r2s = malloc(sizeof(int32_t) * rows);
    uint16_t *recv = malloc(sizeof(uint16_t) * (size_t)rows * H), *out = malloc(sizeof(uint16_t) * (size_t)T * H);
    CK(cudaMemcpy(counts, d_counts, sizeof(int32_t) * E * R, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(t2r, d_t2r, sizeof(int32_t) * rows, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(r2s, d_r2s, sizeof(int32_t) * rows, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(recv, d_recv, sizeof(uint16_t) * (size_t)rows * H, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out, d_out, sizeof(uint16_t) * (size_t)T * H, cudaMemcpyDeviceToHost));

    long total = 0;
    for (int s = 0; s < R; ++s) {
        long per_rank = 0;
        for (int e = 0; e < E; ++e) per_rank += counts[e * R + s];
        REQUIRE(per_rank == (long)B[s] * K, "rank %d: %ld copies, expected %ld", s, per_rank, (long)B[s] * K);
        total += per_rank;
    }
    REQUIRE(total == rows, "%ld copies in all, expected %d", total, rows);
    for (int i = 0; i < rows; ++i) {
        REQUIRE(t2r[i] >= 0 && t2r[i] < rows && r2s[t2r[i]] == i, "maps are not inverse at copy %d", i);
        REQUIRE(memcmp(recv + (size_t)t2r[i] * H, x + (size_t)(i / K) * H, sizeof(uint16_t) * H) == 0,
                "row of copy %d is not its token", i);
    }
    for (int i = 0; i < T * H; ++i) {
        const float want = bf16_value(x[i]), got = bf16_value(out[i]);
        REQUIRE(fabsf(got - want) <= fabsf(want) * 0x1p-7f, "out[%d] = %g, token value %g", i, got, want);
    }
    printf("c abi roundtrip ok: T=%d, %d copies\n", T, rows);
    return 0;
}
