/* A plain C11 client of the kvx C-ABI: two requests pushed layer by layer between two small pools,
 * checked byte by byte on the host, plus the error path of a block id out of range. Built and run
 * by tests/test_c_abi.py; exits 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvx.h"

enum { L = 2, P = 2, H = 2, D = 64, E = 2, BS = 16, NB = 64 };

static int fails = 0;

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "check failed: " __VA_ARGS__); \
            fprintf(stderr, "\n");                        \
            ++fails;                                      \
        }                                                 \
    } while (0)

static uint8_t src_byte(int buf, int64_t off) { return (uint8_t)((off * 131 + buf * 29 + 7) & 0xff); }

int main(void) {
    const size_t row = (size_t)H * D * E, buf_bytes = (size_t)NB * BS * row;
    void *src[L * P], *dst[L * P];
    uint8_t *host = (uint8_t *)malloc(buf_bytes);
    for (int b = 0; b < L * P; ++b) {
        if (cudaMalloc(&src[b], buf_bytes) != cudaSuccess || cudaMalloc(&dst[b], buf_bytes) != cudaSuccess) {
            fprintf(stderr, "cudaMalloc failed\n");
            return 2;
        }
        for (size_t i = 0; i < buf_bytes; ++i) host[i] = src_byte(b, (int64_t)i);
        cudaMemcpy(src[b], host, buf_bytes, cudaMemcpyHostToDevice);
        cudaMemset(dst[b], 0xAB, buf_bytes);
    }
    const kvx_pool sp = {L, P, 1, H, D, E, BS, KVX_LAYOUT_NHD, NB, src};
    const kvx_pool dp = {L, P, 1, H, D, E, BS, KVX_LAYOUT_NHD, NB, dst};
    const int32_t s0[] = {3, 4, 5}, d0[] = {10, 20, 21};   /* 40 tokens: 2 full blocks and 8 rows */
    const int32_t s1[] = {7}, d1[] = {0};                  /* 16 tokens: one block */
    const kvx_request reqs[] = {{100, 40, s0, 3, d0, 3}, {101, 16, s1, 1, d1, 1}};

    kvx_plan_t plan = NULL;
    kvx_status st = kvx_plan(&sp, &dp, reqs, 2, &plan);
    CHECK(st == KVX_OK, "kvx_plan: %s (%s)", kvx_status_str(st), kvx_last_error());
    cudaStream_t stream;
    cudaStreamCreate(&stream);
    for (int l = 0; l < L && st == KVX_OK; ++l) {
        st = kvx_push_layer(plan, l, stream, NULL);
        CHECK(st == KVX_OK, "kvx_push_layer(%d): %s", l, kvx_status_str(st));
    }
    st = kvx_sync(plan, -1);
    CHECK(st == KVX_OK, "kvx_sync: %s (%s)", kvx_status_str(st), kvx_last_error());
    int32_t states[L];
    CHECK(kvx_plan_layer_states(plan, states, L) == KVX_OK, "kvx_plan_layer_states");
    for (int l = 0; l < L; ++l) CHECK(states[l] == KVX_LAYER_DONE, "layer %d state %d", l, states[l]);
    kvx_plan_destroy(plan);

    /* every consumer byte: the producer byte the request maps to it, or the untouched 0xAB */
    for (int b = 0; b < L * P; ++b) {
        cudaMemcpy(host, dst[b], buf_bytes, cudaMemcpyDeviceToHost);
        size_t bad = 0;
        for (int64_t blk = 0; blk < NB; ++blk)
            for (int64_t slot = 0; slot < BS; ++slot) {
                int64_t src_row = -1;
                if (blk == 10 || blk == 20 || (blk == 21 && slot < 8)) {
                    const int64_t t = (blk == 10 ? 0 : blk == 20 ? 16 : 32) + slot;
                    src_row = (int64_t)s0[t / BS] * BS + t % BS;
                } else if (blk == 0) {
                    src_row = (int64_t)s1[0] * BS + slot;
                }
                const uint8_t *got = host + (size_t)(blk * BS + slot) * row;
                for (size_t k = 0; k < row; ++k) {
                    const uint8_t want = src_row < 0 ? 0xAB : src_byte(b, src_row * (int64_t)row + (int64_t)k);
                    bad += got[k] != want;
                }
            }
        CHECK(bad == 0, "buffer %d: %zu bytes differ", b, bad);
    }

    /* the error path: an id outside the pool is refused before any launch, with a reason */
    const int32_t bad_ids[] = {NB};
    const kvx_request bad_req[] = {{1, 4, bad_ids, 1, d1, 1}};
    plan = NULL;
    st = kvx_plan(&sp, &dp, bad_req, 1, &plan);
    CHECK(st == KVX_ERANGE && plan == NULL && strlen(kvx_last_error()) > 0, "out-of-range id: %s",
          kvx_status_str(st));

    for (int b = 0; b < L * P; ++b) {
        cudaFree(src[b]);
        cudaFree(dst[b]);
    }
    cudaStreamDestroy(stream);
    free(host);
    if (fails) return 1;
    printf("c demo ok: %s\n", kvx_version());
    return 0;
}
