/*
 * c_latency.c -- per-call latency of moe_permute and moe_unpermute as a C
 * caller sees it: device memory from the CUDA runtime, calls straight through
 * the C ABI (include/moe_permute.h), no Python.  The benchmark builds and runs
 * it for the small-batch points (T = 1), where a call is bound by launch and
 * latency rather than by HBM bandwidth.
 *
 * usage: moe_c_latency H E E_local K dtype scale_cols T iters
 *   dtype: a moe_dtype_t value (0 = bf16, 2 = fp8 e4m3); E_local < E adds an
 *   expert map with E_local local experts.
 * Prints one JSON object with, for each of permute and unpermute (median
 * over `iters` calls, microseconds):
 *   issue_us   host wall-clock per call of back-to-back calls (what the call
 *              costs the calling thread; the GPU runs behind it);
 *   sync_us    host wall-clock of one call plus cudaStreamSynchronize, after
 *              an idle gap of about 50 us (what a caller that waits for the
 *              result sees end to end);
 *   device_us  CUDA-event time around one call on the stream, after the same
 *              idle gap (the GPU's own latency of the call).
 * and, as the floor every call pays on this machine, the same three figures
 * for moe_permute with num_tokens = 0, which enqueues one tiny kernel
 * (launch_floor_*_us).
 */
#define _POSIX_C_SOURCE 199309L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime_api.h>

#include "moe_permute.h"

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

static uint64_t rng = 0x9e3779b97f4a7c15ull;

static uint32_t next_u32(void)
{
    rng ^= rng >> 12;
    rng ^= rng << 25;
    rng ^= rng >> 27;
    return (uint32_t)((rng * 2685821657736338717ull) >> 32);
}

static double now_us(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec * 1e6 + (double)ts.tv_nsec * 1e-3;
}

static void idle_gap(double us)
{
    double t0 = now_us();
    while (now_us() - t0 < us) {
    }
}

static int cmp_double(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

static double median(double *v, int n)
{
    qsort(v, (size_t)n, sizeof(double), cmp_double);
    return n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
}

struct problem {
    int64_t H, T;
    int32_t E, E_local, K;
    moe_dtype_t dtype;
    int64_t scale_cols;
    void *hidden, *ph, *rows, *out, *ws;
    float *scales, *ps, *w;
    int32_t *ids, *emap, *pidx, *inv;
    int64_t *offsets;
    size_t ws_bytes;
    cudaStream_t s;
};

static void do_permute(struct problem *p)
{
    CHECK_MOE(moe_permute(p->hidden, p->dtype, p->scales, p->scale_cols, p->ids,
                          MOE_INDEX_INT32, p->emap, p->T, p->H, p->K, p->E, p->E_local,
                          p->ph, p->ps, p->offsets, p->pidx, p->inv, p->ws, p->ws_bytes,
                          (moe_stream_t)p->s));
}

static void do_empty_permute(struct problem *p)
{
    CHECK_MOE(moe_permute(NULL, p->dtype, NULL, 0, NULL, MOE_INDEX_INT32, p->emap, 0, p->H, p->K,
                          p->E, p->E_local, NULL, NULL, p->offsets, NULL, NULL, NULL, 0,
                          (moe_stream_t)p->s));
}

static void do_unpermute(struct problem *p)
{
    CHECK_MOE(moe_unpermute(p->rows, p->T * p->K, p->w, p->inv, p->T, p->H, p->K, p->out,
                            p->ws, (moe_stream_t)p->s));
}

static void measure(struct problem *p, void (*fn)(struct problem *), int iters,
                    double *issue_us, double *sync_us, double *device_us)
{
    double *v = (double *)malloc(sizeof(double) * (size_t)iters);
    cudaEvent_t a, b;
    CHECK_CUDA(cudaEventCreate(&a));
    CHECK_CUDA(cudaEventCreate(&b));
    for (int i = 0; i < 100; ++i)
        fn(p);
    CHECK_CUDA(cudaStreamSynchronize(p->s));
    /* back-to-back issue, in rounds of 50 calls so the launch queue never fills */
    int rounds = iters / 50 > 0 ? iters / 50 : 1;
    for (int r = 0; r < rounds; ++r) {
        double t0 = now_us();
        for (int i = 0; i < 50; ++i)
            fn(p);
        v[r] = (now_us() - t0) / 50.0;
        CHECK_CUDA(cudaStreamSynchronize(p->s));
    }
    *issue_us = median(v, rounds);
    for (int i = 0; i < iters; ++i) {
        idle_gap(50.0);
        double t0 = now_us();
        fn(p);
        CHECK_CUDA(cudaStreamSynchronize(p->s));
        v[i] = now_us() - t0;
    }
    *sync_us = median(v, iters);
    for (int i = 0; i < iters; ++i) {
        idle_gap(50.0);
        CHECK_CUDA(cudaEventRecord(a, p->s));
        fn(p);
        CHECK_CUDA(cudaEventRecord(b, p->s));
        CHECK_CUDA(cudaEventSynchronize(b));
        float ms = 0.f;
        CHECK_CUDA(cudaEventElapsedTime(&ms, a, b));
        v[i] = 1e3 * (double)ms;
    }
    *device_us = median(v, iters);
    CHECK_CUDA(cudaEventDestroy(a));
    CHECK_CUDA(cudaEventDestroy(b));
    free(v);
}

static void *dev_alloc(size_t bytes)
{
    void *d = NULL;
    CHECK_CUDA(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    return d;
}

int main(int argc, char **argv)
{
    if (argc != 9) {
        fprintf(stderr, "usage: %s H E E_local K dtype scale_cols T iters\n", argv[0]);
        return 1;
    }
    struct problem p;
    memset(&p, 0, sizeof p);
    p.H = atoll(argv[1]);
    p.E = atoi(argv[2]);
    p.E_local = atoi(argv[3]);
    p.K = atoi(argv[4]);
    p.dtype = (moe_dtype_t)atoi(argv[5]);
    p.scale_cols = atoll(argv[6]);
    p.T = atoll(argv[7]);
    int iters = atoi(argv[8]);
    if (p.H < 1 || p.E < 1 || p.E_local < 1 || p.E_local > p.E || p.K < 1 || p.K > p.E ||
        p.T < 1 || iters < 1 || p.scale_cols < 0)
        return 1;
    const int64_t elem = p.dtype == MOE_DTYPE_FP8_E4M3 ? 1 : 2;
    const int64_t R = p.T * p.K;
    CHECK_CUDA(cudaSetDevice(0));
    CHECK_CUDA(cudaStreamCreateWithFlags(&p.s, cudaStreamNonBlocking));

    /* host inputs: K distinct experts per token; rows of small finite values */
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *emap = (int32_t *)malloc(sizeof(int32_t) * (size_t)p.E);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)p.E);
    for (int64_t t = 0; t < p.T; ++t) {
        for (int32_t e = 0; e < p.E; ++e)
            perm[e] = e;
        for (int32_t k = 0; k < p.K; ++k) {
            int32_t j = k + (int32_t)(next_u32() % (uint32_t)(p.E - k));
            int32_t tmp = perm[k];
            perm[k] = perm[j];
            perm[j] = tmp;
            ids[t * p.K + k] = perm[k];
        }
    }
    for (int32_t e = 0; e < p.E; ++e)
        emap[e] = e < p.E_local ? e : -1;
    size_t hb = (size_t)(p.T * p.H * elem), rb = (size_t)(R * p.H * 2);
    unsigned char *hbytes = (unsigned char *)malloc(hb > rb ? hb : rb);
    for (size_t i = 0; i < (hb > rb ? hb : rb); ++i)
        hbytes[i] = (unsigned char)(0x30 + (next_u32() & 0x0f)); /* finite in every format */
    float *wts = (float *)malloc(sizeof(float) * (size_t)R);
    for (int64_t i = 0; i < R; ++i)
        wts[i] = 1.0f / (float)p.K;

    p.hidden = dev_alloc(hb);
    p.ph = dev_alloc((size_t)(R * p.H * elem));
    p.rows = dev_alloc(rb);
    p.out = dev_alloc((size_t)(p.T * p.H * 2));
    p.ids = (int32_t *)dev_alloc(sizeof(int32_t) * (size_t)R);
    p.pidx = (int32_t *)dev_alloc(sizeof(int32_t) * (size_t)R);
    p.inv = (int32_t *)dev_alloc(sizeof(int32_t) * (size_t)R);
    p.w = (float *)dev_alloc(sizeof(float) * (size_t)R);
    p.offsets = (int64_t *)dev_alloc(sizeof(int64_t) * (size_t)(p.E_local + 1));
    if (p.E_local < p.E) {
        p.emap = (int32_t *)dev_alloc(sizeof(int32_t) * (size_t)p.E);
        CHECK_CUDA(cudaMemcpy(p.emap, emap, sizeof(int32_t) * (size_t)p.E,
                              cudaMemcpyHostToDevice));
    }
    if (p.scale_cols > 0) {
        p.scales = (float *)dev_alloc(sizeof(float) * (size_t)(p.T * p.scale_cols));
        p.ps = (float *)dev_alloc(sizeof(float) * (size_t)(R * p.scale_cols));
        CHECK_CUDA(cudaMemset(p.scales, 0, sizeof(float) * (size_t)(p.T * p.scale_cols)));
    }
    p.ws_bytes = moe_permute_workspace_size(p.T, p.K, p.E);
    p.ws = dev_alloc(p.ws_bytes);
    CHECK_MOE(moe_permute_workspace_init(p.ws, p.ws_bytes, (moe_stream_t)p.s));
    CHECK_CUDA(cudaMemcpy(p.hidden, hbytes, hb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(p.rows, hbytes, rb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(p.ids, ids, sizeof(int32_t) * (size_t)R, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(p.w, wts, sizeof(float) * (size_t)R, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaDeviceSynchronize());

    double pi, ps, pd, ui, us, ud, fi, fs, fd;
    measure(&p, do_permute, iters, &pi, &ps, &pd);
    measure(&p, do_unpermute, iters, &ui, &us, &ud);
    measure(&p, do_empty_permute, iters, &fi, &fs, &fd);
    uint32_t status = 0;
    CHECK_MOE(moe_read_status(p.ws, &status, (moe_stream_t)p.s));
    printf("{\"permute_issue_us\": %.2f, \"permute_sync_us\": %.2f, \"permute_device_us\": %.2f, "
           "\"unpermute_issue_us\": %.2f, \"unpermute_sync_us\": %.2f, "
           "\"unpermute_device_us\": %.2f, \"launch_floor_issue_us\": %.2f, "
           "\"launch_floor_sync_us\": %.2f, \"launch_floor_device_us\": %.2f, "
           "\"status\": %u, \"iters\": %d}\n",
           pi, ps, pd, ui, us, ud, fi, fs, fd, status, iters);
    return status == 0 ? 0 : 4;
}
