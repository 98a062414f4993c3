// Synthetic "prefill" fixture for tests and the benchmark: a bounded integer chain standing in for a
// layer's forward compute on the main stream, optionally followed by a rewrite of that layer's
// producer KV (so a push that ran before the fixture finished would copy stale bytes).
#include "kvx_internal.h"

namespace kvx {

__device__ unsigned long long g_fixture_sink;

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

}  // namespace kvx

using namespace kvx;

extern "C" kvx_status kvx_fixture_prefill(int32_t ctas, int64_t iters, void *buf, int64_t n_bytes, uint64_t seed,
                                          cudaStream_t stream, cudaEvent_t done) {
    if (ctas < 1 || ctas > 65535 || iters < 0) return fail(KVX_EINVAL, "fixture: ctas in [1, 65535], iters >= 0");
    if (buf && (n_bytes < 0 || n_bytes % 16 || ((uintptr_t)buf & 15)))
        return fail(KVX_EINVAL, "fixture: buffer must be 16-byte aligned with a multiple-of-16 size");
    count_launch();
    kvx_fixture_kernel<<<ctas, 128, 0, stream>>>(iters, static_cast<uint4 *>(buf), buf ? n_bytes / 16 : 0, seed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fixture launch");
    if (done) {
        // inside a stream capture the record becomes an event-record node of the graph, so that
        // every replay records `done` where this launch sits
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing(fixture)");
        e = cudaEventRecordWithFlags(done, stream,
                                     cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fixture)");
    }
    return KVX_OK;
}
