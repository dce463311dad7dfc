/*
 * A plain C consumer of the library's C ABI (include/moe_permute.h): device
 * memory from the CUDA runtime, no Python and no torch.  For three seeded
 * problems (one single-launch batch, one routing-grid batch, one batch with an
 * expert map and int64 ids) it runs moe_permute and moe_unpermute and
 * compares every output with the CPU oracle (oracle/moe_oracle.c, linked into
 * this test program) bit for bit.  Prints "ok" and exits 0 on a match.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_permute.h"

/* The oracle's entry points (oracle/moe_oracle.c). */
uint32_t oracle_permute(const void *hidden, int64_t row_bytes, const float *scales,
                        int64_t scale_cols, const void *topk_ids, int ids_are_i64,
                        const int32_t *expert_map, int64_t T, int32_t K, int32_t E,
                        int32_t E_local, int64_t *offsets, int32_t *permuted_idx,
                        int32_t *inv_permuted_idx, void *permuted_hidden, float *permuted_scales);
uint32_t oracle_unpermute(const uint16_t *rows, int64_t num_rows, const float *w,
                          const int32_t *inv, int64_t T, int64_t H, int32_t K, uint16_t *out);

#define CHECK_CUDA(call)                                                             \
    do {                                                                             \
        cudaError_t e_ = (call);                                                     \
        if (e_ != cudaSuccess) {                                                     \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call,             \
                    cudaGetErrorString(e_));                                         \
            exit(2);                                                                 \
        }                                                                            \
    } while (0)

#define CHECK_MOE(call)                                                              \
    do {                                                                             \
        int s_ = (call);                                                             \
        if (s_ != MOE_OK) {                                                          \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call,             \
                    moe_status_string(s_));                                          \
            exit(3);                                                                 \
        }                                                                            \
    } while (0)

static uint64_t rng_state;

static uint32_t next_u32(void)
{
    /* xorshift64* */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (uint32_t)((rng_state * 2685821657736338717ull) >> 32);
}

/* A finite bf16 bit pattern of moderate magnitude (exponent field 0x70..0x8f). */
static uint16_t finite_bf16(void)
{
    uint32_t r = next_u32();
    uint16_t sign = (uint16_t)((r >> 31) << 15);
    uint16_t expo = (uint16_t)(0x70 + ((r >> 7) & 0x1f));
    return (uint16_t)(sign | (expo << 7) | (r & 0x7f));
}

static void *dev_copy(const void *host, size_t bytes)
{
    void *d = NULL;
    CHECK_CUDA(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    if (bytes > 0) CHECK_CUDA(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
    return d;
}

static int same(const char *what, const void *a, const void *b, size_t bytes)
{
    if (memcmp(a, b, bytes) == 0) return 1;
    fprintf(stderr, "mismatch: %s\n", what);
    return 0;
}

/* One problem; returns 1 when every output matches the oracle. */
static int run_case(int64_t T, int32_t K, int32_t E, int32_t E_local, int with_map,
                    int ids64, int64_t H, uint64_t seed)
{
    const int64_t R = T * K;
    const int64_t row_bytes = H * 2;
    rng_state = seed * 0x9E3779B97F4A7C15ull + 1;

    uint16_t *hidden = malloc((size_t)(T * H) * 2);
    uint16_t *rows = malloc((size_t)(R * H) * 2);
    float *w = malloc((size_t)R * sizeof(float));
    int32_t *ids32 = malloc((size_t)R * 4);
    int64_t *ids64v = malloc((size_t)R * 8);
    int32_t *map = malloc((size_t)E * 4);
    for (int64_t i = 0; i < T * H; ++i) hidden[i] = finite_bf16();
    for (int64_t i = 0; i < R * H; ++i) rows[i] = finite_bf16();
    for (int64_t i = 0; i < R; ++i) w[i] = (float)(next_u32() >> 8) / 16777216.0f;
    for (int64_t i = 0; i < R; ++i) {
        ids32[i] = (int32_t)(next_u32() % (uint32_t)E);
        ids64v[i] = ids32[i];
    }
    /* map: every fourth global expert is local, numbered in order; the rest -1 */
    for (int32_t e = 0; e < E; ++e) map[e] = (e % 4 == 0 && e / 4 < E_local) ? e / 4 : -1;
    const void *ids_host = ids64 ? (const void *)ids64v : (const void *)ids32;

    /* oracle */
    int64_t *r_off = malloc((size_t)(E_local + 1) * 8);
    int32_t *r_pidx = malloc((size_t)R * 4), *r_inv = malloc((size_t)R * 4);
    uint16_t *r_ph = calloc((size_t)(R * H), 2);
    uint16_t *r_out = malloc((size_t)(T * H) * 2);
    uint32_t r_flags = oracle_permute(hidden, row_bytes, NULL, 0, ids_host, ids64,
                                      with_map ? map : NULL, T, K, E, E_local, r_off, r_pidx,
                                      r_inv, r_ph, NULL);
    oracle_unpermute(rows, R, w, r_inv, T, H, K, r_out);

    /* library */
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    void *d_hidden = dev_copy(hidden, (size_t)(T * H) * 2);
    void *d_rows = dev_copy(rows, (size_t)(R * H) * 2);
    float *d_w = dev_copy(w, (size_t)R * 4);
    void *d_ids = dev_copy(ids_host, (size_t)R * (ids64 ? 8 : 4));
    int32_t *d_map = with_map ? dev_copy(map, (size_t)E * 4) : NULL;
    int64_t *d_off;
    int32_t *d_pidx, *d_inv;
    void *d_ph, *d_out, *d_ws;
    CHECK_CUDA(cudaMalloc((void **)&d_off, (size_t)(E_local + 1) * 8));
    CHECK_CUDA(cudaMalloc((void **)&d_pidx, (size_t)R * 4));
    CHECK_CUDA(cudaMalloc((void **)&d_inv, (size_t)R * 4));
    CHECK_CUDA(cudaMalloc(&d_ph, (size_t)(R * H) * 2));
    CHECK_CUDA(cudaMalloc(&d_out, (size_t)(T * H) * 2));
    size_t ws_bytes = moe_permute_workspace_size(T, K, E);
    if (ws_bytes == 0) {
        fprintf(stderr, "workspace size query failed\n");
        return 0;
    }
    CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    CHECK_MOE(moe_permute_workspace_init(d_ws, ws_bytes, stream));
    CHECK_MOE(moe_permute(d_hidden, MOE_DTYPE_BF16, NULL, 0, d_ids,
                          ids64 ? MOE_INDEX_INT64 : MOE_INDEX_INT32, d_map, T, H, K, E, E_local,
                          d_ph, NULL, d_off, d_pidx, d_inv, d_ws, ws_bytes, stream));
    CHECK_MOE(moe_unpermute(d_rows, R, d_w, d_inv, T, H, K, d_out, d_ws, stream));
    uint32_t status = 0;
    CHECK_MOE(moe_read_status(d_ws, &status, stream));  /* synchronises the stream */

    int64_t *g_off = malloc((size_t)(E_local + 1) * 8);
    int32_t *g_pidx = malloc((size_t)R * 4), *g_inv = malloc((size_t)R * 4);
    uint16_t *g_ph = malloc((size_t)(R * H) * 2);
    uint16_t *g_out = malloc((size_t)(T * H) * 2);
    CHECK_CUDA(cudaMemcpy(g_off, d_off, (size_t)(E_local + 1) * 8, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(g_pidx, d_pidx, (size_t)R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(g_inv, d_inv, (size_t)R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(g_ph, d_ph, (size_t)(R * H) * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(g_out, d_out, (size_t)(T * H) * 2, cudaMemcpyDeviceToHost));

    int ok = 1;
    const int64_t n_valid = r_off[E_local];
    ok &= status == r_flags;
    if (status != r_flags) fprintf(stderr, "status %u, oracle flags %u\n", status, r_flags);
    ok &= same("expert_first_token_offset", g_off, r_off, (size_t)(E_local + 1) * 8);
    ok &= same("permuted_idx", g_pidx, r_pidx, (size_t)R * 4);
    ok &= same("inv_permuted_idx", g_inv, r_inv, (size_t)R * 4);
    ok &= same("permuted rows", g_ph, r_ph, (size_t)(n_valid * H) * 2);
    ok &= same("unpermute output", g_out, r_out, (size_t)(T * H) * 2);
    printf("T=%lld K=%d E=%d E_local=%d map=%d ids64=%d H=%lld kept rows=%lld: %s\n",
           (long long)T, K, E, E_local, with_map, ids64, (long long)H, (long long)n_valid,
           ok ? "match" : "MISMATCH");

    cudaFree(d_hidden); cudaFree(d_rows); cudaFree(d_w); cudaFree(d_ids);
    if (d_map) cudaFree(d_map);
    cudaFree(d_off); cudaFree(d_pidx); cudaFree(d_inv); cudaFree(d_ph); cudaFree(d_out);
    cudaFree(d_ws);
    cudaStreamDestroy(stream);
    free(hidden); free(rows); free(w); free(ids32); free(ids64v); free(map);
    free(r_off); free(r_pidx); free(r_inv); free(r_ph); free(r_out);
    free(g_off); free(g_pidx); free(g_inv); free(g_ph); free(g_out);
    return ok;
}

int main(void)
{
    int dev = 0;
    CHECK_CUDA(cudaGetDevice(&dev));
    if (moe_permute_supported(dev) != 1) {
        fprintf(stderr, "device %d is not supported by this library\n", dev);
        return 4;
    }
    int ok = 1;
    ok &= run_case(100, 2, 8, 8, 0, 0, 256, 1);     /* 200 rows: single launch */
    ok &= run_case(3000, 2, 8, 8, 0, 0, 256, 2);    /* routing grid + gather */
    ok &= run_case(2500, 6, 64, 16, 1, 1, 512, 3);  /* expert map, int64 ids */
    if (!ok) return 1;
    printf("ok\n");
    return 0;
}
