// Synthetic "prefill" fixture for the kvx tests and benchmark: a bounded integer chain standing in
// for a layer's forward compute on the main stream, optionally followed by a rewrite of that layer's
// producer KV (so a push that ran before the fixture finished would copy stale bytes). Built into
// its own library; the kvx library does not contain it.
#include "kvx_fixture.h"
#include "kvx.h"

#include <atomic>
#include <chrono>
#include <cstdio>
#include <deque>
#include <vector>

namespace {

__device__ unsigned long long g_fixture_sink;

std::atomic<int64_t> g_launches{0};
thread_local char g_error[256];

int fixture_fail(const char *what) {
    std::snprintf(g_error, sizeof(g_error), "%s", what);
    return -1;
}

int fixture_cuda_fail(cudaError_t e, const char *what) {
    std::snprintf(g_error, sizeof(g_error), "%s: %s", what, cudaGetErrorString(e));
    return -1;
}

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void __launch_bounds__(128) kvx_fixture_kernel(int64_t iters, uint4 *buf, int64_t n_vec, uint64_t seed) {
    uint64_t x = seed ^ (uint64_t)(blockIdx.x * blockDim.x + threadIdx.x);
    for (int64_t i = 0; i < iters; ++i) x = x * 6364136223846793005ull + 1442695040888963407ull;
    if (x == 0x0123456789ABCDEFull) atomicAdd(&g_fixture_sink, 1ull);   // keeps the chain live
    if (buf) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += (int64_t)gridDim.x * blockDim.x) {
            const uint64_t a = splitmix64(seed * 0x100000001B3ull + 2 * (uint64_t)i);
            const uint64_t b = splitmix64(seed * 0x100000001B3ull + 2 * (uint64_t)i + 1);
            buf[i] = make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
        }
    }
}

}  // namespace

extern "C" int kvx_fixture_prefill(int32_t ctas, int64_t iters, void *buf, int64_t n_bytes, uint64_t seed,
                                   cudaStream_t stream, cudaEvent_t done) {
    if (ctas < 1 || ctas > 65535 || iters < 0) return fixture_fail("fixture: ctas in [1, 65535], iters >= 0");
    if (buf && (n_bytes < 0 || n_bytes % 16 || ((uintptr_t)buf & 15)))
        return fixture_fail("fixture: buffer must be 16-byte aligned with a multiple-of-16 size");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    kvx_fixture_kernel<<<ctas, 128, 0, stream>>>(iters, static_cast<uint4 *>(buf), buf ? n_bytes / 16 : 0, seed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fixture_cuda_fail(e, "fixture launch");
    if (done) {
        // inside a stream capture the record becomes an event-record node of the graph, so that
        // every replay records `done` where this launch sits
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return fixture_cuda_fail(e, "cudaStreamIsCapturing(fixture)");
        e = cudaEventRecordWithFlags(done, stream,
                                     cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
        if (e != cudaSuccess) return fixture_cuda_fail(e, "cudaEventRecord(fixture)");
    }
    return 0;
}

extern "C" int64_t kvx_fixture_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char *kvx_fixture_last_error(void) { return g_error; }

namespace {

double us_since(std::chrono::steady_clock::time_point t0) {
    return std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
}

int kvx_fail(const char *what, kvx_status st) {
    std::snprintf(g_error, sizeof(g_error), "%s: %s: %s", what, kvx_status_str(st), kvx_last_error());
    return -1;
}

struct Issued {
    kvx_plan_t plan = nullptr;
    bool timed = false;
};

}  // namespace

extern "C" int kvx_fixture_run_steps(const kvx_pool *src, const kvx_pool *dst, const kvx_request *reqs,
                                     int32_t n_reqs, const kvx_plan_opts *opts, int32_t every, int32_t n_steps,
                                     int32_t all_layers, int32_t fixture_ctas, int64_t fixture_iters,
                                     cudaStream_t main, cudaStream_t side, const cudaEvent_t *ready,
                                     const cudaEvent_t *marks, int64_t *start_ns, int64_t *end_ns, int64_t cap,
                                     int64_t *n_stamps, double *issue_us, double *plan_us, int32_t lookahead) {
    if (!src || !dst || !ready || n_steps < 0 || every < 1 || lookahead < 1)
        return fixture_fail("run_steps: bad arguments");
    const int32_t n_layers = src->n_layers;
    kvx_plan_opts plain{}, timing{};
    if (opts) plain = *opts;
    timing = plain;
    timing.flags |= KVX_PLAN_TIMING;
    if (n_stamps) *n_stamps = 0;
    std::vector<int64_t> s_ns(4096), e_ns(4096);

    // syncs a step's plan, keeps its stamps when it was timed, destroys it
    auto finish = [&](const Issued &p) -> int {
        kvx_status st = kvx_sync(p.plan, -1);
        if (st != KVX_OK) { kvx_plan_destroy(p.plan); return kvx_fail("kvx_sync", st); }
        if (p.timed && start_ns && end_ns && n_stamps) {
            int32_t n = 0;
            st = kvx_plan_push_times_ns(p.plan, s_ns.data(), e_ns.data(), (int32_t)s_ns.size(), &n);
            if (st != KVX_OK) { kvx_plan_destroy(p.plan); return kvx_fail("kvx_plan_push_times_ns", st); }
            for (int32_t k = 0; k < n && *n_stamps < cap; ++k, ++*n_stamps) {
                start_ns[*n_stamps] = s_ns[k];
                end_ns[*n_stamps] = e_ns[k];
            }
        }
        kvx_status d = kvx_plan_destroy(p.plan);
        return d == KVX_OK ? 0 : kvx_fail("kvx_plan_destroy", d);
    };

    std::deque<Issued> inflight;   // issued steps not yet synced, oldest first
    auto drain = [&](size_t keep) -> int {
        while (inflight.size() > keep) {
            const Issued p = inflight.front();
            inflight.pop_front();
            if (finish(p)) {
                for (const Issued &q : inflight) kvx_plan_destroy(q.plan);
                inflight.clear();
                return -1;
            }
        }
        return 0;
    };
    for (int32_t i = 0; i < n_steps; ++i) {
        const auto h0 = std::chrono::steady_clock::now();
        if (marks && cudaEventRecord(marks[i], main) != cudaSuccess) return fixture_fail("run_steps: mark record");
        Issued cur;
        cur.timed = i % every == 0;
        kvx_status st = kvx_plan_ex(src, dst, reqs, n_reqs, cur.timed ? &timing : &plain, &cur.plan);
        if (st != KVX_OK) return kvx_fail("kvx_plan_ex", st);
        if (plan_us) plan_us[i] = us_since(h0);
        for (int32_t l = 0; l < n_layers; ++l) {
            if (kvx_fixture_prefill(fixture_ctas, fixture_iters, nullptr, 0, (uint64_t)l, main, ready[l])) return -1;
            if (!all_layers) {
                st = kvx_push_layer(cur.plan, l, side, ready[l]);
                if (st != KVX_OK) return kvx_fail("kvx_push_layer", st);
            }
        }
        if (all_layers) {
            st = kvx_push_layers(cur.plan, 0, n_layers, side, ready[n_layers - 1]);
            if (st != KVX_OK) return kvx_fail("kvx_push_layers", st);
        }
        if (issue_us) issue_us[i] = us_since(h0);
        inflight.push_back(cur);
        if (drain((size_t)lookahead)) return -1;
    }
    if (drain(0)) return -1;
    if (marks && cudaEventRecord(marks[n_steps], main) != cudaSuccess) return fixture_fail("run_steps: mark record");
    return 0;
}
