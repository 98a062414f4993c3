// The layer push: a tile-table driven gather/scatter copy kernel for sm_103a, the side-stream issue
// path, completion counting and per-layer status.
//
// Follows the push-mode NIXL connector article (spke.com 3844), "Implementierungsdetails" step 3
// (write the KV blocks into the consumer's memory, one completion per write, the consumer counts
// them) and "Threading-Modell" (issue off the main loop), and the "vLLM MoRIIO KV Connector" notes,
// section 3.2 (per-layer writes gated by a CUDA event, sealed write count) and section 6 (per-layer
// DONE / FAILED / PENDING batch state).
#include "kvx_internal.h"

#include <chrono>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>

namespace kvx {

// ------------------------------------------------------------------------------------------------
// Copy kernel
// ------------------------------------------------------------------------------------------------

template <int VEC> struct VecType;
template <> struct VecType<16> { using T = uint4; };
template <> struct VecType<8> { using T = uint2; };
template <> struct VecType<4> { using T = uint32_t; };
template <> struct VecType<2> { using T = uint16_t; };
template <> struct VecType<1> { using T = uint8_t; };

constexpr int kUnroll = 4;

// One CTA per (tile, plane, layer). Every thread reads the 32-byte tile descriptor (a broadcast
// load), resolves the (layer, plane, shard) buffer bases, then copies with VEC-byte integer vectors,
// kUnroll independent loads in flight per thread before their stores. Values are never converted.
template <int VEC, bool STRIDED>
__global__ void __launch_bounds__(1024) kvx_copy_tiles(CopyArgs a) {
    using V = typename VecType<VEC>::T;
    const TileDesc t = a.tiles[blockIdx.x];
    const int32_t layer = a.layer0 + (int32_t)blockIdx.z;
    const int64_t lp = (int64_t)layer * a.n_planes + blockIdx.y;

    // Bounds guard: host-built tables are validated already; device-built ones are checked here.
    // An out-of-bounds tile sets the layer's error word and is skipped (no trap).
    const int64_t src_end = STRIDED ? t.src_off + (int64_t)(t.n - 1) * a.src_pitch + a.width : t.src_off + t.n;
    const int64_t dst_end = STRIDED ? t.dst_off + (int64_t)(t.n - 1) * a.dst_pitch + a.width : t.dst_off + t.n;
    if (t.n <= 0 || t.src_off < 0 || t.dst_off < 0 || src_end > a.src_buf_bytes || dst_end > a.dst_buf_bytes ||
        t.s_shard < 0 || t.s_shard >= a.src_shards || t.d_shard < 0 || t.d_shard >= a.dst_shards) {
        if (threadIdx.x == 0 && t.n != 0) atomicOr(&a.err[layer], 1);
        return;
    }
    const uint8_t *src = a.src_base[lp * a.src_shards + t.s_shard] + t.src_off;
    uint8_t *dst = a.dst_base[lp * a.dst_shards + t.d_shard] + t.dst_off;

    if (!STRIDED) {
        const V *s = reinterpret_cast<const V *>(src);
        V *d = reinterpret_cast<V *>(dst);
        const int32_t nv = t.n / VEC;
        const int32_t step = (int32_t)blockDim.x;
        for (int32_t i = threadIdx.x; i < nv; i += step * kUnroll) {
            V r[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i + u * step < nv) r[u] = s[i + u * step];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i + u * step < nv) d[i + u * step] = r[u];
        }
    } else {
        // Rows of `width` bytes at the two pitches. Threads are laid out as (row lane, column) once,
        // so the loop has no per-element division.
        const int32_t vpr = a.width / VEC;
        if (vpr <= (int32_t)blockDim.x) {
            const int32_t rpp = (int32_t)blockDim.x / vpr;          // rows per pass
            const int32_t my_row = (int32_t)threadIdx.x / vpr;
            const int32_t col = (int32_t)threadIdx.x - my_row * vpr;
            if (my_row < rpp) {
                for (int32_t row = my_row; row < t.n; row += rpp * kUnroll) {
                    V r[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int32_t rr = row + u * rpp;
                        if (rr < t.n) r[u] = reinterpret_cast<const V *>(src + (int64_t)rr * a.src_pitch)[col];
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int32_t rr = row + u * rpp;
                        if (rr < t.n) reinterpret_cast<V *>(dst + (int64_t)rr * a.dst_pitch)[col] = r[u];
                    }
                }
            }
        } else {
            for (int32_t row = 0; row < t.n; ++row) {
                const V *s = reinterpret_cast<const V *>(src + (int64_t)row * a.src_pitch);
                V *d = reinterpret_cast<V *>(dst + (int64_t)row * a.dst_pitch);
                for (int32_t c = threadIdx.x; c < vpr; c += blockDim.x) d[c] = s[c];
            }
        }
    }
}

template <int VEC>
static cudaError_t launch_vec(const CopyArgs &a, dim3 grid, int threads, bool strided, cudaStream_t st) {
    if (strided)
        kvx_copy_tiles<VEC, true><<<grid, threads, 0, st>>>(a);
    else
        kvx_copy_tiles<VEC, false><<<grid, threads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_copy(const CopyArgs &a, int64_t n_tiles, int32_t n_layers, int32_t vec, bool strided,
                        int32_t threads, cudaStream_t st) {
    if (n_tiles <= 0 || n_layers <= 0) return cudaSuccess;
    const dim3 grid((unsigned)n_tiles, (unsigned)a.n_planes, (unsigned)n_layers);
    count_launch();
    switch (vec) {
        case 16: return launch_vec<16>(a, grid, threads, strided, st);
        case 8: return launch_vec<8>(a, grid, threads, strided, st);
        case 4: return launch_vec<4>(a, grid, threads, strided, st);
        case 2: return launch_vec<2>(a, grid, threads, strided, st);
        default: return launch_vec<1>(a, grid, threads, strided, st);
    }
}

// ------------------------------------------------------------------------------------------------
// Device memory pool and auxiliary stream
// ------------------------------------------------------------------------------------------------

static std::mutex g_dev_mu;
static std::map<int, cudaMemPool_t> g_pools;
static std::map<int, cudaStream_t> g_aux;

static cudaError_t device_pool(int dev, cudaMemPool_t *out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_pools.find(dev);
    if (it != g_pools.end()) { *out = it->second; return cudaSuccess; }
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;   // keep freed blocks for reuse (plans may be rebuilt every step)
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    g_pools[dev] = pool;
    *out = pool;
    return cudaSuccess;
}

kvx_status pool_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaMemPool_t pool;
    e = device_pool(dev, &pool);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    e = cudaMallocFromPoolAsync(ptr, bytes < 256 ? 256 : bytes, pool, stream);
    if (e == cudaErrorMemoryAllocation) return fail(KVX_ENOMEM, "device allocation of %zu bytes failed", bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync");
    return KVX_OK;
}

// Callers guarantee no work that uses ptr is still pending, so any stream may order the free.
void pool_free(void *ptr) {
    if (ptr) cudaFreeAsync(ptr, cudaStreamPerThread);
}

// kvx_sync reads status words here, so it never waits behind work the caller queued on its own
// streams after the pushes.
kvx_status aux_stream(cudaStream_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_aux.find(dev);
    if (it == g_aux.end()) {
        cudaStream_t s;
        e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate(aux)");
        it = g_aux.emplace(dev, s).first;
    }
    *out = it->second;
    return KVX_OK;
}

void plan_layout(kvx_plan_s *pl) {
    const size_t a = 256;
    pl->off_tiles = 0;
    pl->off_src = align_up(sizeof(TileDesc) * (size_t)pl->n_tiles, a);
    pl->off_dst = pl->off_src + align_up(sizeof(void *) * pl->src_base.size(), a);
    pl->off_err = pl->off_dst + align_up(sizeof(void *) * pl->dst_base.size(), a);
    pl->dev_bytes = pl->off_err + align_up(sizeof(int32_t) * (size_t)pl->src.n_layers, a);
}

CopyArgs plan_copy_args(const kvx_plan_s *pl, int32_t layer0) {
    CopyArgs a;
    uint8_t *base = static_cast<uint8_t *>(pl->dev);
    a.tiles = reinterpret_cast<const TileDesc *>(base + pl->off_tiles);
    a.src_base = reinterpret_cast<const uint8_t *const *>(base + pl->off_src);
    a.dst_base = reinterpret_cast<uint8_t *const *>(base + pl->off_dst);
    a.err = reinterpret_cast<int32_t *>(base + pl->off_err);
    a.src_buf_bytes = pl->src.buf_bytes();
    a.dst_buf_bytes = pl->dst.buf_bytes();
    a.src_pitch = pl->src.row_bytes();
    a.dst_pitch = pl->dst.row_bytes();
    a.width = pl->width;
    a.n_planes = pl->src.n_planes;
    a.src_shards = pl->src.n_shards;
    a.dst_shards = pl->dst.n_shards;
    a.layer0 = layer0;
    return a;
}

}  // namespace kvx

using namespace kvx;

// ------------------------------------------------------------------------------------------------
// Plan upload, push, sync
// ------------------------------------------------------------------------------------------------

// Allocates and uploads a host-built plan's descriptors on `stream` (first push only); later pushes
// on other streams wait for the upload.
static kvx_status ensure_device(kvx_plan_s *pl, cudaStream_t stream) {
    if (pl->uploaded) {
        if (stream != pl->upload_stream) {
            cudaError_t e = cudaStreamWaitEvent(stream, pl->upload_evt, 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(upload)");
        }
        return KVX_OK;
    }
    plan_layout(pl);
    kvx_status st = pool_alloc(&pl->dev, pl->dev_bytes, stream);
    if (st) return st;
    // one host image of the descriptor block, uploaded with a single copy; the plan keeps the image
    // until it is destroyed, so the copy never reads freed host memory
    pl->upload_img.assign(pl->dev_bytes, 0);
    uint8_t *img = pl->upload_img.data();
    if (pl->n_tiles) memcpy(img + pl->off_tiles, pl->tiles.data(), sizeof(TileDesc) * (size_t)pl->n_tiles);
    memcpy(img + pl->off_src, pl->src_base.data(), sizeof(void *) * pl->src_base.size());
    memcpy(img + pl->off_dst, pl->dst_base.data(), sizeof(void *) * pl->dst_base.size());
    cudaError_t e = cudaMemcpyAsync(pl->dev, img, pl->dev_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(plan upload)");
    e = cudaEventCreateWithFlags(&pl->upload_evt, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    e = cudaEventRecord(pl->upload_evt, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(upload)");
    pl->upload_stream = stream;
    pl->uploaded = true;
    return KVX_OK;
}

// Timing plans use timing-enabled events for both ends of a push; other plans only need completion.
static kvx_status take_event(kvx_plan_s *pl, cudaEvent_t *ev) {
    if (!pl->free_events.empty()) {
        *ev = pl->free_events.back();
        pl->free_events.pop_back();
        return KVX_OK;
    }
    const unsigned flags = (pl->flags & KVX_PLAN_TIMING) ? cudaEventDefault : cudaEventDisableTiming;
    cudaError_t e = cudaEventCreateWithFlags(ev, flags);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    return KVX_OK;
}

extern "C" {

kvx_status kvx_push_layers(kvx_plan_t pl, int32_t l0, int32_t l1, cudaStream_t stream, cudaEvent_t ready) {
    if (!pl) return fail(KVX_EINVAL, "NULL plan");
    if (l0 < 0 || l1 > pl->src.n_layers || l0 >= l1)
        return fail(KVX_EINVAL, "layer range [%d, %d) outside [0, %d)", l0, l1, pl->src.n_layers);
    kvx_status st = ensure_device(pl, stream);
    if (st) return st;
    cudaError_t e;
    if (ready) {
        e = cudaStreamWaitEvent(stream, ready, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(ready)");
    }
    cudaEvent_t start = nullptr;
    if (pl->flags & KVX_PLAN_TIMING) {
        st = take_event(pl, &start);
        if (st) return st;
        e = cudaEventRecord(start, stream);
        if (e != cudaSuccess) {
            pl->free_events.push_back(start);
            return cuda_fail(e, "cudaEventRecord(push start)");
        }
    }
    e = launch_copy(plan_copy_args(pl, l0), pl->n_tiles, l1 - l0, pl->vec, pl->strided != 0, pl->threads, stream);
    if (e != cudaSuccess) {
        if (start) pl->free_events.push_back(start);
        for (int32_t l = l0; l < l1; ++l) pl->layer_state[l] = KVX_LAYER_FAILED;
        return cuda_fail(e, "copy kernel launch");
    }
    cudaEvent_t ev;
    st = take_event(pl, &ev);
    if (st) return st;
    e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) {
        pl->free_events.push_back(ev);
        if (start) pl->free_events.push_back(start);
        return cuda_fail(e, "cudaEventRecord(push)");
    }
    pl->pending.push_back({ev, start, l0, l1});
    for (int32_t l = l0; l < l1; ++l) {
        pl->layer_state[l] = KVX_LAYER_PENDING;
        if (pl->inject[l]) { pl->injected_pending[l] = 1; pl->inject[l] = 0; }
    }
    return KVX_OK;
}

kvx_status kvx_push_layer(kvx_plan_t pl, int32_t layer, cudaStream_t stream, cudaEvent_t ready) {
    return kvx_push_layers(pl, layer, layer + 1, stream, ready);
}

kvx_status kvx_sync(kvx_plan_t pl, int64_t timeout_us) {
    if (!pl) return fail(KVX_EINVAL, "NULL plan");
    const size_t sealed = pl->pending.size();   // pushes issued so far
    if (sealed == 0) {
        for (int32_t s : pl->layer_state)
            if (s == KVX_LAYER_FAILED) return fail(KVX_EFAILED, "a layer reported FAILED");
        return KVX_OK;
    }
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::microseconds(timeout_us < 0 ? 0 : timeout_us);
    for (size_t i = 0; i < sealed; ++i) {
        cudaEvent_t ev = pl->pending[i].done;
        if (timeout_us < 0) {
            cudaError_t e = cudaEventSynchronize(ev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize(push)");
            continue;
        }
        for (;;) {
            cudaError_t e = cudaEventQuery(ev);
            if (e == cudaSuccess) break;
            if (e != cudaErrorNotReady) return cuda_fail(e, "cudaEventQuery(push)");
            if (std::chrono::steady_clock::now() >= deadline)
                return fail(KVX_ETIMEDOUT, "%zu of %zu pushes still pending at the deadline", sealed - i, sealed);
            std::this_thread::yield();
        }
    }
    // every sealed push finished: read the per-layer error words the kernels may have set
    std::vector<int32_t> err((size_t)pl->src.n_layers, 0);
    cudaStream_t aux = nullptr;
    kvx_status ast = aux_stream(&aux);
    if (ast) return ast;
    int32_t *d_err = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(pl->dev) + pl->off_err);
    cudaError_t e = cudaMemcpyAsync(err.data(), d_err, sizeof(int32_t) * err.size(), cudaMemcpyDeviceToHost, aux);
    if (e == cudaSuccess) e = cudaStreamSynchronize(aux);
    if (e != cudaSuccess) return cuda_fail(e, "reading push error words");
    bool any_err = false;
    for (int32_t v : err) any_err |= (v != 0);
    if (any_err) {
        e = cudaMemsetAsync(d_err, 0, sizeof(int32_t) * err.size(), aux);
        if (e == cudaSuccess) e = cudaStreamSynchronize(aux);
        if (e != cudaSuccess) return cuda_fail(e, "clearing push error words");
    }
    bool failed = false;
    pl->push_us.clear();
    for (size_t i = 0; i < sealed; ++i) {
        const PendingPush &p = pl->pending[i];
        if (p.start) {
            float ms = 0.f;
            e = cudaEventElapsedTime(&ms, p.start, p.done);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime(push)");
            pl->push_us.push_back(ms * 1000.f);
            pl->free_events.push_back(p.start);
        }
        for (int32_t l = p.layer_begin; l < p.layer_end; ++l) {
            const bool bad = err[l] != 0 || pl->injected_pending[l];
            pl->layer_state[l] = bad ? KVX_LAYER_FAILED : KVX_LAYER_DONE;
            failed |= bad;
        }
        pl->free_events.push_back(p.done);
    }
    for (auto &x : pl->injected_pending) x = 0;
    pl->pending.erase(pl->pending.begin(), pl->pending.begin() + (long)sealed);
    if (failed) return fail(KVX_EFAILED, "at least one layer reported FAILED");
    return KVX_OK;
}

kvx_status kvx_plan_destroy(kvx_plan_t pl) {
    if (!pl) return KVX_OK;
    kvx_status st = KVX_OK;
    for (const PendingPush &p : pl->pending) {
        cudaError_t e = cudaEventSynchronize(p.done);
        if (e != cudaSuccess && st == KVX_OK) st = cuda_fail(e, "cudaEventSynchronize(destroy)");
        cudaEventDestroy(p.done);
        if (p.start) cudaEventDestroy(p.start);
    }
    for (cudaEvent_t ev : pl->free_events) cudaEventDestroy(ev);
    if (pl->upload_evt) {
        cudaEventSynchronize(pl->upload_evt);
        cudaEventDestroy(pl->upload_evt);
    }
    if (pl->dev) pool_free(pl->dev);
    delete pl;
    return st;
}

}  // extern "C"
