/* Requests per second through the host connector's whole protocol, called from C (no binding
 * between): registration and the last prefill chunk (alternate requests in the other order, so half
 * go through DEFERRED), poll (READY), start, one queued write, seal, its report (every layer DONE),
 * poll (DONE), release. The connector makes no CUDA call, so no GPU is needed. Usage:
 *     kvx_conn_rate [n_requests]
 * Prints "requests_per_s <rate>" and exits 0 when every request reached DONE. Built and run by
 * tests/test_c_abi.py. */
#define _POSIX_C_SOURCE 199309L   /* clock_gettime under -std=c11 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

#include "kvx.h"

static double now_s(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

int main(int argc, char **argv) {
    const int64_t n = argc > 1 ? atoll(argv[1]) : 200000;
    int32_t ids[16], states[64];
    for (int i = 0; i < 16; ++i) ids[i] = i;
    for (int i = 0; i < 64; ++i) states[i] = KVX_LAYER_DONE;
    kvx_conn_t conn = NULL;
    if (kvx_conn_create(NULL, &conn) != KVX_OK) {
        fprintf(stderr, "kvx_conn_create: %s\n", kvx_last_error());
        return 2;
    }
    kvx_conn_event ev[8];
    int32_t n_ev = 0;
    int64_t done = 0, bad = 0;
    const double t0 = now_s();
    for (int64_t r = 0; r < n; ++r) {
        kvx_status st = KVX_OK;
        if (r & 1) {
            st |= kvx_conn_prefill(conn, r, 0, ids, 16, 256, 1, r);
            st |= kvx_conn_register(conn, r, 0, ids, 16, r);
        } else {
            st |= kvx_conn_register(conn, r, 0, ids, 16, r);
            st |= kvx_conn_prefill(conn, r, 0, ids, 16, 256, 1, r);
        }
        st |= kvx_conn_poll(conn, r, ev, 8, &n_ev);
        st |= kvx_conn_start(conn, r, 0, r);
        st |= kvx_conn_write_issued(conn, r, 0, 0, 1);
        st |= kvx_conn_seal(conn, r, 0, 0);
        st |= kvx_conn_write_done(conn, r, 0, 0, states, 64, NULL, 0, r);
        st |= kvx_conn_poll(conn, r, ev, 8, &n_ev);
        for (int32_t i = 0; i < n_ev; ++i) done += ev[i].req_id == r && ev[i].state == KVX_CONN_DONE;
        st |= kvx_conn_release(conn, r);
        bad += st != KVX_OK;
    }
    const double dt = now_s() - t0;
    kvx_conn_destroy(conn);
    printf("requests_per_s %.1f\n", (double)n / dt);
    if (bad || done != n) {
        fprintf(stderr, "%lld calls failed, %lld of %lld requests reached DONE\n", (long long)bad, (long long)done,
                (long long)n);
        return 1;
    }
    return 0;
}
