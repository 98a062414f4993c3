/*
 * Synthetic prefill fixture for the kvx tests and benchmark. Not part of the kvx library or its
 * C-ABI: it is built into its own library (libkvx_fixture.so) and stands in for a layer's forward
 * compute on the caller's main stream, so that layer pushes can be gated on a layer's ready event.
 */
#ifndef KVX_FIXTURE_H
#define KVX_FIXTURE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Occupies `ctas` CTAs of 128 threads with a dependent integer chain of `iters` steps per thread.
 * If `buf` is not NULL, the CTAs then rewrite buf[0 .. n_bytes) (device, 16-byte aligned, n_bytes a
 * multiple of 16) with a pattern derived from `seed`, so a push that ran before the fixture finished
 * would copy stale bytes. `done`, when not NULL, is recorded right after the kernel. May be called
 * while `stream` is being captured into a CUDA graph: `done` is then recorded by an external
 * event-record node on every replay (the launch counter counts the capture only).
 * Returns 0, or -1 with a reason in kvx_fixture_last_error() (ctas outside [1, 65535], iters < 0,
 * a misaligned buffer, a failed CUDA call).
 */
int kvx_fixture_prefill(int32_t ctas, int64_t iters, void *buf, int64_t n_bytes, uint64_t seed,
                        cudaStream_t stream, cudaEvent_t done);

/*
 * The benchmark's engine loop, in native code (the issuing loop of a serving engine is native; a
 * Python loop of ctypes calls is slower than the GPU work it issues). Runs n_steps steps through the
 * kvx C-ABI. Step i: kvx_plan_ex(src, dst, reqs, opts) -- with KVX_PLAN_TIMING added when
 * i % every == 0 -- then per layer l: the fixture (fixture_ctas CTAs x fixture_iters) on `main`,
 * ready[l] recorded after it, and kvx_push_layer(plan, l, side, ready[l]) (with all_layers != 0: the
 * fixtures of every layer, then one kvx_push_layers over all of them gated on the last layer's
 * event). A step's plan is synced (kvx_sync, no deadline) once `lookahead` later steps have been
 * issued (1: after the next one), then destroyed; the last ones after the loop. marks, when not NULL, holds n_steps + 1 events: marks[i] is recorded on `main` where
 * step i starts, marks[n_steps] after the last step's sync. The timed plans' push stamps (global
 * timer, ns) are appended to start_ns / end_ns (up to cap entries; *n_stamps receives the count);
 * issue_us[i] / plan_us[i] (may be NULL) receive the host time to issue step i and to build its
 * plan. Returns 0, or -1 with a reason in kvx_fixture_last_error().
 */
struct kvx_pool;
struct kvx_request;
struct kvx_plan_opts;
int kvx_fixture_run_steps(const struct kvx_pool *src, const struct kvx_pool *dst, const struct kvx_request *reqs,
                          int32_t n_reqs, const struct kvx_plan_opts *opts, int32_t every, int32_t n_steps,
                          int32_t all_layers, int32_t fixture_ctas, int64_t fixture_iters, cudaStream_t main,
                          cudaStream_t side, const cudaEvent_t *ready, const cudaEvent_t *marks, int64_t *start_ns,
                          int64_t *end_ns, int64_t cap, int64_t *n_stamps, double *issue_us, double *plan_us,
                          int32_t lookahead);

/* Fixture kernels launched by this process so far. */
int64_t kvx_fixture_launch_count(void);

/* Reason for the calling thread's last failed call. */
const char *kvx_fixture_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVX_FIXTURE_H */
