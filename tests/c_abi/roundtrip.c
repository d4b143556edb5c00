/*
 * A plain C caller of the library's C ABI (include/kvc.h): create a cache
 * over device pools, claim blocks from the FIFO pool, map positions to slots,
 * append K/V rows, run paged GQA decode attention, and check the result
 * against a host computation of softmax(q K^T * scale) V done in double
 * precision straight from the appended rows in position order (no block
 * table, no slots).
 *
 * Build: cc roundtrip.c -I<repo>/include -I<cuda>/include -L<lib dir> -lkvc -lcudart
 * Exit status 0 and a line "c_abi_roundtrip ok" on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvc.h"

enum { L = 1, NB = 12, BS = 16, HKV = 2, HQ = 6, D = 64, B = 3, MAXB = 7 };
static const int CTX[B] = {1, 40, 100}; /* blocks: 1, 3, 7 -> 11 of the 12 */

#define CHECK(call)                                                                      \
    do {                                                                                 \
        kvc_status st_ = (call);                                                         \
        if (st_ != KVC_OK) {                                                             \
            fprintf(stderr, "%s failed: %d (%s)\n", #call, (int)st_, kvc_last_error_string()); \
            return 1;                                                                    \
        }                                                                                \
    } while (0)
#define CUDA(call)                                                                       \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));           \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

static uint32_t lcg_state = 12345u;
/* a multiple of 2^-10 in [-1, 1]: exactly representable in binary16 */
static float draw(void) {
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return (float)((int)(lcg_state >> 8) % 2049 - 1024) / 1024.0f;
}

/* binary16 bits of a value that binary16 represents exactly (normal or zero), by its definition:
 * sign, 5-bit exponent with bias 15, 10 fraction bits */
static uint16_t to_half_exact(float x) {
    if (x == 0.0f) return 0;
    uint16_t sign = x < 0 ? 0x8000u : 0;
    int e;
    double m = frexp(fabs((double)x), &e); /* |x| = m * 2^e, m in [0.5, 1) */
    int exp16 = e - 1 + 15;                /* |x| = (2m) * 2^(e-1) */
    uint32_t frac = (uint32_t)((2.0 * m - 1.0) * 1024.0);
    return (uint16_t)(sign | (uint16_t)(exp16 << 10) | (uint16_t)frac);
}

int main(void) {
    kvc_config cfg = {L, NB, BS, HKV, D, KVC_F16};
    size_t pool_bytes = 0;
    CHECK(kv_cache_pool_bytes(&cfg, &pool_bytes));
    if (pool_bytes != (size_t)L * NB * HKV * BS * D * 2) {
        fprintf(stderr, "pool bytes %zu\n", pool_bytes);
        return 1;
    }
    void *k_pool = NULL, *v_pool = NULL;
    CUDA(cudaMalloc(&k_pool, pool_bytes));
    CUDA(cudaMalloc(&v_pool, pool_bytes));
    kvc_handle h = NULL;
    CHECK(kv_cache_create(&cfg, k_pool, v_pool, &h));

    /* scatter the physical blocks: claim all, give them back in a shuffled order, claim again (FIFO) */
    int32_t ids[NB];
    for (int i = 0; i < NB; ++i) CHECK(kv_block_alloc(h, &ids[i]));
    const int order[NB] = {7, 2, 11, 0, 9, 4, 1, 10, 5, 3, 8, 6};
    for (int i = 0; i < NB; ++i) CHECK(kv_block_release(h, ids[order[i]]));
    int32_t table[B][MAXB];
    memset(table, 0, sizeof(table));
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < (CTX[b] + BS - 1) / BS; ++j) CHECK(kv_block_alloc(h, &table[b][j]));
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < (CTX[b] + BS - 1) / BS; ++j)
            if (table[b][j] != ids[order[(b == 0 ? 0 : b == 1 ? 1 : 4) + j]]) {
                fprintf(stderr, "FIFO order broken at sequence %d block %d\n", b, j);
                return 1;
            }
    double util = 0;
    CHECK(kv_cache_utilisation(h, &util));
    if (fabs(util - 100.0 * 11 / NB) > 1e-9) {
        fprintf(stderr, "utilisation %f\n", util);
        return 1;
    }

    /* every position of every sequence, packed in order; its slot from the library's slot arithmetic */
    int n = 0, first[B], count[B];
    for (int b = 0; b < B; ++b) {
        first[b] = 0;
        count[b] = CTX[b];
        n += CTX[b];
    }
    int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * n);
    CHECK(kv_slot_mapping(&table[0][0], MAXB, B, first, count, BS, slots));
    float* kf = (float*)malloc(sizeof(float) * n * HKV * D);
    float* vf = (float*)malloc(sizeof(float) * n * HKV * D);
    uint16_t* kh = (uint16_t*)malloc(2 * (size_t)n * HKV * D);
    uint16_t* vh = (uint16_t*)malloc(2 * (size_t)n * HKV * D);
    for (int i = 0; i < n * HKV * D; ++i) {
        kf[i] = draw();
        vf[i] = draw();
        kh[i] = to_half_exact(kf[i]);
        vh[i] = to_half_exact(vf[i]);
    }
    float qf[B * HQ * D];
    uint16_t qh[B * HQ * D];
    for (int i = 0; i < B * HQ * D; ++i) {
        qf[i] = draw();
        qh[i] = to_half_exact(qf[i]);
    }
    void *dk, *dv, *dslots, *dq, *dtable, *dctx, *dout;
    CUDA(cudaMalloc(&dk, 2 * (size_t)n * HKV * D));
    CUDA(cudaMalloc(&dv, 2 * (size_t)n * HKV * D));
    CUDA(cudaMalloc(&dslots, sizeof(int64_t) * n));
    CUDA(cudaMalloc(&dq, sizeof(qh)));
    CUDA(cudaMalloc(&dtable, sizeof(table)));
    CUDA(cudaMalloc(&dctx, sizeof(CTX)));
    CUDA(cudaMalloc(&dout, sizeof(float) * B * HQ * D));
    CUDA(cudaMemcpy(dk, kh, 2 * (size_t)n * HKV * D, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dv, vh, 2 * (size_t)n * HKV * D, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dslots, slots, sizeof(int64_t) * n, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dq, qh, sizeof(qh), cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dtable, table, sizeof(table), cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dctx, CTX, sizeof(CTX), cudaMemcpyHostToDevice));

    CHECK(kv_append(h, 0, dk, dv, (const int64_t*)dslots, n, NULL));
    int nsplit = 0, bps = 0;
    size_t ws_bytes = 0;
    CHECK(paged_decode_plan(B, HQ, HKV, D, BS, 100, 0, &nsplit, &bps, &ws_bytes));
    void* ws = NULL;
    if (ws_bytes) CUDA(cudaMalloc(&ws, ws_bytes));
    void *kl = NULL, *vl = NULL;
    CHECK(kv_cache_layer(h, 0, &kl, &vl));
    const float scale = 0.125f;
    CHECK(paged_decode_attention(dq, kl, vl, NB, (const int32_t*)dtable, MAXB, (const int32_t*)dctx, B, HQ, HKV, D,
                                 BS, 100, scale, dout, KVC_F32, ws, ws_bytes, 0, NULL));
    float out[B * HQ * D];
    CUDA(cudaMemcpy(out, dout, sizeof(out), cudaMemcpyDeviceToHost));
    uint32_t flags = 1;
    CHECK(kvc_device_error_flags(&flags, 1));
    if (flags != 0) {
        fprintf(stderr, "device error flags 0x%x\n", flags);
        return 1;
    }

    /* host check: rows in position order, softmax in double */
    double max_err = 0;
    int row0 = 0;
    for (int b = 0; b < B; ++b) {
        for (int hq = 0; hq < HQ; ++hq) {
            const int hk = hq / (HQ / HKV);
            double s[100], m = -INFINITY, l = 0;
            for (int j = 0; j < CTX[b]; ++j) {
                double dot = 0;
                for (int c = 0; c < D; ++c)
                    dot += (double)qf[(b * HQ + hq) * D + c] * kf[((size_t)(row0 + j) * HKV + hk) * D + c];
                s[j] = dot * scale;
                if (s[j] > m) m = s[j];
            }
            for (int j = 0; j < CTX[b]; ++j) l += exp(s[j] - m);
            for (int c = 0; c < D; ++c) {
                double o = 0;
                for (int j = 0; j < CTX[b]; ++j) o += exp(s[j] - m) * vf[((size_t)(row0 + j) * HKV + hk) * D + c];
                const double err = fabs(o / l - out[(b * HQ + hq) * D + c]);
                if (!(err <= max_err)) max_err = err; /* NaN propagates */
            }
        }
        row0 += CTX[b];
    }
    CHECK(kv_cache_destroy(h));
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dslots);
    cudaFree(dq);
    cudaFree(dtable);
    cudaFree(dctx);
    cudaFree(dout);
    cudaFree(ws);
    cudaFree(k_pool);
    cudaFree(v_pool);
    free(slots);
    free(kf);
    free(vf);
    free(kh);
    free(vh);
    if (!(max_err <= 2e-3)) {
        fprintf(stderr, "max error %g beyond 2e-3\n", max_err);
        return 1;
    }
    printf("c_abi_roundtrip ok max_err=%.3g\n", max_err);
    return 0;
}
