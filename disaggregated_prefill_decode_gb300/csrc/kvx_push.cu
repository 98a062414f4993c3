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
#include <algorithm>
#include <map>
#include <tuple>
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

// Host-validated tables never fail this guard; device-built ones are checked here. An out-of-bounds
// tile is skipped and its layer's error word set (no trap).
template <bool STRIDED>
__device__ __forceinline__ bool tile_in_bounds(const TileDesc &t, const CopyArgs &a) {
    const int64_t src_end = STRIDED ? t.src_off + (int64_t)(t.n - 1) * a.src_pitch + a.width : t.src_off + t.n;
    const int64_t dst_end = STRIDED ? t.dst_off + (int64_t)(t.n - 1) * a.dst_pitch + a.width : t.dst_off + t.n;
    return t.n > 0 && t.src_off >= 0 && t.dst_off >= 0 && src_end <= a.src_buf_bytes && dst_end <= a.dst_buf_bytes &&
           t.s_shard >= 0 && t.s_shard < a.src_shards && t.d_shard >= 0 && t.d_shard < a.dst_shards;
}

// Copies one tile with VEC-byte integer vectors, kUnroll independent loads in flight per thread
// before their stores. Values are never converted.
template <int VEC, bool STRIDED>
__device__ __forceinline__ void copy_tile(const TileDesc &t, const uint8_t *src, uint8_t *dst, const CopyArgs &a) {
    using V = typename VecType<VEC>::T;
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Timing plans: every CTA folds the device's global timer into its push's slot when it starts
// (minimum) and when it is done (maximum), so a slot ends up holding the span from the first CTA's
// start to the last CTA's end. One clock serves the whole GPU; no host call is involved.
__device__ __forceinline__ void stamp_start(const CopyArgs &a) {
    if (a.ts_start && threadIdx.x == 0) atomicMin(a.ts_start, (unsigned long long)global_ns());
}

// Called by every thread of the CTA (the test on a kernel argument is uniform). Each thread's stores
// are made visible device-wide before the stamp, so the span covers them.
__device__ __forceinline__ void stamp_end(const CopyArgs &a) {
    if (!a.ts_end) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(a.ts_end, (unsigned long long)global_ns());
}

// Work item w of a launch: tile w % n_tiles of plane (w / n_tiles) % n_planes of layer
// layer0 + w / (n_tiles * n_planes). Consecutive items are consecutive tiles of one buffer pair.
__device__ __forceinline__ void decode_item(const CopyArgs &a, int64_t w, int64_t *tile, int32_t *layer, int64_t *lp) {
    const int64_t rest = w / a.n_tiles;
    *tile = w - rest * a.n_tiles;
    const int32_t plane = (int32_t)(rest % a.n_planes);
    *layer = a.layer0 + (int32_t)(rest / a.n_planes);
    *lp = (int64_t)(*layer) * a.n_planes + plane;
}

// KVX_KERNEL_TILE: one CTA per (tile, plane, layer).
template <int VEC, bool STRIDED>
__global__ void __launch_bounds__(1024) kvx_copy_tiles(CopyArgs a) {
    stamp_start(a);
    const TileDesc t = a.tiles[blockIdx.x];
    const int32_t layer = a.layer0 + (int32_t)blockIdx.z;
    const int64_t lp = (int64_t)layer * a.n_planes + blockIdx.y;
    if (!tile_in_bounds<STRIDED>(t, a)) {
        if (threadIdx.x == 0 && t.n != 0) atomicOr(&a.err[layer], 1);
    } else {
        copy_tile<VEC, STRIDED>(t, a.src_base[lp * a.src_shards + t.s_shard] + t.src_off,
                                a.dst_base[lp * a.dst_shards + t.d_shard] + t.dst_off, a);
    }
    stamp_end(a);
}

// KVX_KERNEL_PERSIST: a resident grid walks the work items; each CTA loads the next item's
// descriptor before copying the current one, so the descriptor latency hides behind the copy.
template <int VEC, bool STRIDED>
__global__ void __launch_bounds__(1024) kvx_copy_persist(CopyArgs a, int64_t n_work) {
    int64_t w = blockIdx.x;
    if (w >= n_work) return;
    stamp_start(a);
    TileDesc next = a.tiles[w % a.n_tiles];
    for (; w < n_work; w += gridDim.x) {
        const TileDesc t = next;
        if (w + gridDim.x < n_work) next = a.tiles[(w + gridDim.x) % a.n_tiles];
        int64_t tile, lp;
        int32_t layer;
        decode_item(a, w, &tile, &layer, &lp);
        if (!tile_in_bounds<STRIDED>(t, a)) {
            if (threadIdx.x == 0 && t.n != 0) atomicOr(&a.err[layer], 1);
            continue;
        }
        copy_tile<VEC, STRIDED>(t, a.src_base[lp * a.src_shards + t.s_shard] + t.src_off,
                                a.dst_base[lp * a.dst_shards + t.d_shard] + t.dst_off, a);
    }
    stamp_end(a);
}

// ------------------------------------------------------------------------------------------------
// KVX_KERNEL_BULK: bulk asynchronous copies through shared memory (16-byte aligned).
// One thread per CTA drives a ring of STAGES stages: the load of an item lands in its stage
// and completes the stage's mbarrier (transaction count = bytes); the thread then issues the bulk
// store of that stage and, once the store before it has finished reading its stage, the load of a
// later item into that freed stage. Waits are bounded by the global timer.
// A strided tile (rows of `width` bytes at each side's pitch) is packed densely in its stage: a side
// whose pitch equals the width moves in one bulk copy, the other side row by row, all rows of a
// load completing on the stage's one mbarrier and all row stores forming one bulk group.
// ------------------------------------------------------------------------------------------------

constexpr uint64_t kBulkWaitNs = 2000000000ull;   // 2 s: far beyond any legitimate tile copy

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

// The single arrival of a stage's phase, announcing `bytes` of incoming transactions (0 for none).
__device__ __forceinline__ void mbar_arrive_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for a stage's phase; false when the deadline passed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > kBulkWaitNs) return false;
    return true;
}

__device__ __forceinline__ void bulk_load(void *stage, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(stage)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *stage, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(stage)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

struct BulkItem {
    const uint8_t *src;
    uint8_t *dst;
    uint32_t bytes;    // 0: skipped (out of bounds or misaligned)
    int32_t rows;      // strided tiles: rows of a.width bytes; contiguous tiles: 1
    int32_t layer;
};

template <bool STRIDED>
__device__ __forceinline__ BulkItem bulk_item(const CopyArgs &a, int64_t w, int32_t stage_bytes) {
    int64_t tile, lp;
    BulkItem it;
    decode_item(a, w, &tile, &it.layer, &lp);
    const TileDesc t = a.tiles[tile];
    it.src = nullptr;
    it.dst = nullptr;
    it.bytes = 0;
    it.rows = STRIDED ? t.n : 1;
    const int64_t bytes = STRIDED ? (int64_t)t.n * a.width : (int64_t)t.n;
    if (!tile_in_bounds<STRIDED>(t, a) || bytes > stage_bytes) {
        if (t.n != 0) atomicOr(&a.err[it.layer], 1);
        return it;
    }
    it.src = a.src_base[lp * a.src_shards + t.s_shard] + t.src_off;
    it.dst = a.dst_base[lp * a.dst_shards + t.d_shard] + t.dst_off;
    uintptr_t mis = ((uintptr_t)it.src) | ((uintptr_t)it.dst) | (uintptr_t)bytes;
    if (STRIDED) mis |= (uintptr_t)a.width | (uintptr_t)a.src_pitch | (uintptr_t)a.dst_pitch;
    if (mis & 15) {
        atomicOr(&a.err[it.layer], 1);
        return it;
    }
    it.bytes = (uint32_t)bytes;
    return it;
}

template <int STAGES, bool STRIDED>
__global__ void __launch_bounds__(32) kvx_copy_bulk(CopyArgs a, int64_t n_work, int32_t stage_bytes) {
    constexpr int kBulkStages = STAGES;
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bar[kBulkStages];
    if (threadIdx.x != 0) return;
    stamp_start(a);
    for (int s = 0; s < kBulkStages; ++s) mbar_init(&bar[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    const int64_t n_mine = (int64_t)blockIdx.x < n_work ? (n_work - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    BulkItem items[kBulkStages];
    // item i of this CTA is work item blockIdx.x + i * gridDim.x, in stage i % kBulkStages
    const bool src_packed = !STRIDED || a.src_pitch == a.width;    // one bulk copy per tile on that side
    const bool dst_packed = !STRIDED || a.dst_pitch == a.width;
    auto issue = [&](int64_t i) {
        const int s = (int)(i % kBulkStages);
        const BulkItem it = bulk_item<STRIDED>(a, blockIdx.x + i * gridDim.x, stage_bytes);
        items[s] = it;
        mbar_arrive_expect(&bar[s], it.bytes);
        if (!it.bytes) return;
        uint8_t *stage = ring + (size_t)s * stage_bytes;
        if (src_packed) {
            bulk_load(stage, it.src, it.bytes, &bar[s]);
        } else {
            for (int32_t r = 0; r < it.rows; ++r)
                bulk_load(stage + (size_t)r * a.width, it.src + (int64_t)r * a.src_pitch, (uint32_t)a.width, &bar[s]);
        }
    };
    int64_t issued = 0;
    for (; issued < n_mine && issued < kBulkStages - 1; ++issued) issue(issued);
    bool timed_out = false;
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = (int)(i % kBulkStages);
        if (!mbar_wait(&bar[s], (uint32_t)((i / kBulkStages) & 1))) {
            atomicOr(&a.err[items[s].layer], 2);
            timed_out = true;
            break;
        }
        if (items[s].bytes) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint8_t *stage = ring + (size_t)s * stage_bytes;
            if (dst_packed) {
                bulk_store(items[s].dst, stage, items[s].bytes);
            } else {
                for (int32_t r = 0; r < items[s].rows; ++r)
                    bulk_store(items[s].dst + (int64_t)r * a.dst_pitch, stage + (size_t)r * a.width, (uint32_t)a.width);
            }
        }
        bulk_commit();
        if (issued < n_mine) {
            bulk_wait_read_1();   // the stores issued one item ago have read the stage the next load reuses
            issue(issued);
            ++issued;
        }
    }
    if (timed_out) {
        // give every load still in flight a bounded chance to land before the ring goes away
        for (int64_t j = 0; j < kBulkStages && j < issued; ++j) {
            const int64_t i = issued - 1 - j;
            mbar_wait(&bar[i % kBulkStages], (uint32_t)((i / kBulkStages) & 1));
        }
    }
    bulk_wait_all();   // the stores have completed, not only read their stages
    if (a.ts_end) atomicMax(a.ts_end, (unsigned long long)global_ns());
}

// ------------------------------------------------------------------------------------------------
// Launch
// ------------------------------------------------------------------------------------------------

template <int VEC>
static cudaError_t launch_vec(const CopyArgs &a, int32_t n_layers, const LaunchShape &sh, unsigned grid_persist,
                              cudaStream_t st) {
    const int64_t n_work = a.n_tiles * a.n_planes * n_layers;
    if (sh.kernel == KVX_KERNEL_TILE) {
        const dim3 grid((unsigned)a.n_tiles, (unsigned)a.n_planes, (unsigned)n_layers);
        if (sh.strided) kvx_copy_tiles<VEC, true><<<grid, sh.threads, 0, st>>>(a);
        else kvx_copy_tiles<VEC, false><<<grid, sh.threads, 0, st>>>(a);
    } else {
        if (sh.strided) kvx_copy_persist<VEC, true><<<grid_persist, sh.threads, 0, st>>>(a, n_work);
        else kvx_copy_persist<VEC, false><<<grid_persist, sh.threads, 0, st>>>(a, n_work);
    }
    return cudaGetLastError();
}

// Resident CTAs per SM for a kernel (occupancy query), times the SM count; cached per key.
static std::mutex g_grid_mu;
static std::map<std::tuple<int, const void *, int, int>, int> g_resident;

static cudaError_t resident_grid(const void *fn, int threads, int smem, int per_sm_cap, int *grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_grid_mu);
    const auto key = std::make_tuple(dev, fn, threads, smem);
    auto it = g_resident.find(key);
    if (it == g_resident.end()) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (smem > 0) {
            // one limit per kernel, large enough for every ring it may be launched with
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkRingMax);
            if (e != cudaSuccess) return e;
        }
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
        if (e != cudaSuccess) return e;
        it = g_resident.emplace(key, sms * 1000 + std::max(per_sm, 1)).first;
    }
    const int sms = it->second / 1000, per_sm = it->second % 1000;
    *grid = sms * (per_sm_cap > 0 ? std::min(per_sm_cap, per_sm) : per_sm);
    return cudaSuccess;
}

template <bool STRIDED>
static const void *bulk_fn_of(int stages) {
    switch (stages) {
        case 2: return (const void *)kvx_copy_bulk<2, STRIDED>;
        case 3: return (const void *)kvx_copy_bulk<3, STRIDED>;
        case 6: return (const void *)kvx_copy_bulk<6, STRIDED>;
        case 8: return (const void *)kvx_copy_bulk<8, STRIDED>;
        default: return (const void *)kvx_copy_bulk<4, STRIDED>;
    }
}

static const void *bulk_fn(int stages, bool strided) {
    return strided ? bulk_fn_of<true>(stages) : bulk_fn_of<false>(stages);
}

template <int VEC>
static const void *persist_fn(bool strided) {
    return strided ? (const void *)kvx_copy_persist<VEC, true> : (const void *)kvx_copy_persist<VEC, false>;
}

cudaError_t launch_copy(const CopyArgs &a, int32_t n_layers, const LaunchShape &sh, cudaStream_t st) {
    if (a.n_tiles <= 0 || n_layers <= 0) return cudaSuccess;
    const int64_t n_work = a.n_tiles * a.n_planes * n_layers;
    count_launch();
    int grid = 0;
    cudaError_t e;
    if (sh.kernel == KVX_KERNEL_BULK) {
        const int smem = sh.stages * sh.tile_bytes;
        const int cap = sh.ctas_per_sm ? sh.ctas_per_sm : (n_work * (int64_t)sh.tile_bytes < ((int64_t)128 << 20) ? 1 : 64);
        const void *fn = bulk_fn(sh.stages, sh.strided != 0);
        e = resident_grid(fn, 32, smem, cap, &grid);
        if (e != cudaSuccess) return e;
        CopyArgs args_copy = a;
        int64_t work = n_work;
        int32_t stage_bytes = sh.tile_bytes;
        void *args[] = {&args_copy, &work, &stage_bytes};
        return cudaLaunchKernel(fn, dim3((unsigned)std::min<int64_t>(grid, n_work)), dim3(32), args, (size_t)smem, st);
    }
    // default resident CTAs: small launches stay small so that they overlap the caller's compute and
    // the next push; large ones take the whole GPU
    LaunchShape shape = sh;
    if (shape.ctas_per_sm == 0) shape.ctas_per_sm = n_work * (int64_t)sh.tile_bytes < ((int64_t)128 << 20) ? 2 : 64;
    if (sh.kernel == KVX_KERNEL_PERSIST) {
        const void *fn = sh.vec == 16 ? persist_fn<16>(sh.strided) : sh.vec == 8 ? persist_fn<8>(sh.strided)
                       : sh.vec == 4 ? persist_fn<4>(sh.strided) : sh.vec == 2 ? persist_fn<2>(sh.strided)
                       : persist_fn<1>(sh.strided);
        e = resident_grid(fn, sh.threads, 0, shape.ctas_per_sm, &grid);
        if (e != cudaSuccess) return e;
        grid = (int)std::min<int64_t>(grid, n_work);
    }
    switch (sh.vec) {
        case 16: return launch_vec<16>(a, n_layers, sh, (unsigned)grid, st);
        case 8: return launch_vec<8>(a, n_layers, sh, (unsigned)grid, st);
        case 4: return launch_vec<4>(a, n_layers, sh, (unsigned)grid, st);
        case 2: return launch_vec<2>(a, n_layers, sh, (unsigned)grid, st);
        default: return launch_vec<1>(a, n_layers, sh, (unsigned)grid, st);
    }
}

// ------------------------------------------------------------------------------------------------
// Device memory pool and auxiliary stream
// ------------------------------------------------------------------------------------------------

static std::mutex g_dev_mu;
static std::map<int, cudaMemPool_t> g_pools;
static std::map<int, cudaStream_t> g_aux;
static std::map<std::pair<int, int>, std::vector<cudaStream_t>> g_lanes;
static std::mutex g_evt_mu;
static std::map<int, std::vector<cudaEvent_t>> g_events;   // per device, timing disabled

kvx_status event_take(cudaEvent_t *ev) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    {
        std::lock_guard<std::mutex> lk(g_evt_mu);
        std::vector<cudaEvent_t> &v = g_events[dev];
        if (!v.empty()) {
            *ev = v.back();
            v.pop_back();
            return KVX_OK;
        }
    }
    e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    return KVX_OK;
}

// Events go back to the pool of the current device; callers give back events of that device.
void event_give(cudaEvent_t ev) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaEventDestroy(ev);
        return;
    }
    std::lock_guard<std::mutex> lk(g_evt_mu);
    g_events[dev].push_back(ev);
}

// Lane `i` for the current device at `priority`: a non-blocking stream created on first use and kept
// for the life of the process.
static kvx_status lane_stream(int32_t i, int priority, cudaStream_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    std::vector<cudaStream_t> &v = g_lanes[std::make_pair(dev, priority)];
    while ((int32_t)v.size() <= i) {
        cudaStream_t s;
        e = cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, priority);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate(lane)");
        v.push_back(s);
    }
    *out = v[i];
    return KVX_OK;
}

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
    a.ts_start = nullptr;
    a.ts_end = nullptr;
    a.n_tiles = pl->n_tiles;
    a.src_buf_bytes = pl->src.buf_bytes();
    a.dst_buf_bytes = pl->dst.buf_bytes();
    a.src_pitch = pl->src_pitch;
    a.dst_pitch = pl->dst_pitch;
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
    st = event_take(&pl->upload_evt);
    if (st) return st;
    e = cudaEventRecord(pl->upload_evt, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(upload)");
    pl->upload_stream = stream;
    pl->uploaded = true;
    return KVX_OK;
}

// Stamp slots of a timing plan: kTimingSlots starts (set to all ones, folded with atomicMin) then
// kTimingSlots ends (zero, folded with atomicMax), allocated and set on `stream` at the first timed push.
static kvx_status reset_timing_slots(kvx_plan_s *pl, int32_t n, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(pl->ts, 0xFF, sizeof(unsigned long long) * (size_t)n, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(pl->ts + kTimingSlots, 0, sizeof(unsigned long long) * (size_t)n, stream);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e, "cudaMemsetAsync(timing slots)");
}

static kvx_status ensure_timing_slots(kvx_plan_s *pl, cudaStream_t stream) {
    if (pl->ts) return KVX_OK;
    void *p = nullptr;
    kvx_status st = pool_alloc(&p, sizeof(unsigned long long) * 2 * (size_t)kTimingSlots, stream);
    if (st) return st;
    pl->ts = static_cast<unsigned long long *>(p);
    return reset_timing_slots(pl, kTimingSlots, stream);
}

// Completion events; timing comes from the kernels' own global-timer stamps.
static kvx_status take_event(kvx_plan_s *pl, cudaEvent_t *ev) {
    if (!pl->free_events.empty()) {
        *ev = pl->free_events.back();
        pl->free_events.pop_back();
        return KVX_OK;
    }
    return event_take(ev);
}

extern "C" {

kvx_status kvx_push_layer_notify(kvx_plan_t pl, int32_t l0, int32_t l1, cudaStream_t stream, cudaEvent_t ready,
                                 cudaEvent_t done) {
    if (!pl) return fail(KVX_EINVAL, "NULL plan");
    if (l0 < 0 || l1 > pl->src.n_layers || l0 >= l1)
        return fail(KVX_EINVAL, "layer range [%d, %d) outside [0, %d)", l0, l1, pl->src.n_layers);
    kvx_status st = ensure_device(pl, stream);
    if (st) return st;
    cudaError_t e;
    // timing plans: the push's global-timer slot (stamps live in a buffer set up on the caller's
    // stream before the fork, so every lane sees it initialised)
    int32_t slot = -1;
    if (pl->flags & KVX_PLAN_TIMING) {
        st = ensure_timing_slots(pl, stream);
        if (st) return st;
        if ((int32_t)pl->pending.size() < kTimingSlots) slot = (int32_t)pl->pending.size();
    }
    if (pl->lanes > 1) {
        // fork: the lane waits for everything already on the caller's stream (the upload included)
        if (!pl->fork_evt) {
            st = event_take(&pl->fork_evt);
            if (st) return st;
        }
        e = cudaEventRecord(pl->fork_evt, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
        if (pl->lane_src != stream || (int32_t)pl->lane_cache.size() != pl->lanes) {
            // first push from this stream: look up its priority and the lanes that match it once
            int prio = 0;
            e = cudaStreamGetPriority(stream, &prio);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetPriority");
            pl->lane_cache.assign(pl->lanes, nullptr);
            for (int32_t i = 0; i < pl->lanes; ++i) {
                st = lane_stream(i, prio, &pl->lane_cache[i]);
                if (st) return st;
            }
            pl->lane_src = stream;
        }
        cudaStream_t lane = pl->lane_cache[pl->next_lane];
        pl->next_lane = (pl->next_lane + 1) % pl->lanes;
        e = cudaStreamWaitEvent(lane, pl->fork_evt, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(fork)");
        stream = lane;
    }
    if (ready) {
        e = cudaStreamWaitEvent(stream, ready, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(ready)");
    }
    const LaunchShape shape{pl->kernel, pl->vec, pl->strided, pl->threads, pl->tile_bytes, pl->ctas_per_sm,
                            pl->bulk_stages};
    CopyArgs args = plan_copy_args(pl, l0);
    if (slot >= 0) {
        args.ts_start = pl->ts + slot;
        args.ts_end = pl->ts + kTimingSlots + slot;
    }
    e = launch_copy(args, l1 - l0, shape, stream);
    if (e != cudaSuccess) {
        for (int32_t l = l0; l < l1; ++l) pl->layer_state[l] = KVX_LAYER_FAILED;
        return cuda_fail(e, "copy kernel launch");
    }
    cudaEvent_t ev;
    st = take_event(pl, &ev);
    if (st) return st;
    e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) {
        pl->free_events.push_back(ev);
        return cuda_fail(e, "cudaEventRecord(push)");
    }
    if (done) {
        e = cudaEventRecord(done, stream);
        if (e != cudaSuccess) {
            pl->free_events.push_back(ev);
            return cuda_fail(e, "cudaEventRecord(done)");
        }
    }
    pl->pending.push_back({ev, slot, l0, l1});
    for (int32_t l = l0; l < l1; ++l) {
        pl->layer_state[l] = KVX_LAYER_PENDING;
        if (pl->inject[l]) { pl->injected_pending[l] = 1; pl->inject[l] = 0; }
    }
    return KVX_OK;
}

kvx_status kvx_push_layers(kvx_plan_t pl, int32_t l0, int32_t l1, cudaStream_t stream, cudaEvent_t ready) {
    return kvx_push_layer_notify(pl, l0, l1, stream, ready, nullptr);
}

kvx_status kvx_push_layer(kvx_plan_t pl, int32_t layer, cudaStream_t stream, cudaEvent_t ready) {
    return kvx_push_layer_notify(pl, layer, layer + 1, stream, ready, nullptr);
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
    pl->push_start_us.clear();
    pl->push_end_us.clear();
    pl->push_start_ns.clear();
    pl->push_end_ns.clear();
    int32_t n_slots = 0;
    for (size_t i = 0; i < sealed; ++i) n_slots = std::max(n_slots, pl->pending[i].slot + 1);
    if (n_slots > 0) {
        // the kernels' global-timer stamps, then fresh slots for the next pushes
        std::vector<unsigned long long> t0((size_t)n_slots), t1((size_t)n_slots);
        e = cudaMemcpyAsync(t0.data(), pl->ts, sizeof(unsigned long long) * t0.size(), cudaMemcpyDeviceToHost, aux);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(t1.data(), pl->ts + kTimingSlots, sizeof(unsigned long long) * t1.size(),
                                cudaMemcpyDeviceToHost, aux);
        if (e != cudaSuccess) return cuda_fail(e, "reading push timing stamps");
        kvx_status rs = reset_timing_slots(pl, n_slots, aux);
        if (rs) return rs;
        e = cudaStreamSynchronize(aux);
        if (e != cudaSuccess) return cuda_fail(e, "reading push timing stamps");
        unsigned long long base = ~0ull;
        for (size_t i = 0; i < sealed; ++i) {
            const int32_t k = pl->pending[i].slot;
            if (k >= 0 && t0[k] != ~0ull) base = std::min(base, t0[k]);
        }
        for (size_t i = 0; i < sealed; ++i) {
            const int32_t k = pl->pending[i].slot;
            if (k < 0 || t0[k] == ~0ull) continue;   // untimed, or a launch with nothing to copy
            pl->push_start_ns.push_back((int64_t)t0[k]);
            pl->push_end_ns.push_back((int64_t)t1[k]);
            pl->push_start_us.push_back((float)((double)(t0[k] - base) * 1e-3));
            pl->push_end_us.push_back((float)((double)(t1[k] - base) * 1e-3));
        }
    }
    for (size_t i = 0; i < sealed; ++i) {
        const PendingPush &p = pl->pending[i];
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
        event_give(p.done);
    }
    for (cudaEvent_t ev : pl->free_events) event_give(ev);
    if (pl->fork_evt) event_give(pl->fork_evt);
    if (pl->upload_evt) {
        cudaEventSynchronize(pl->upload_evt);
        event_give(pl->upload_evt);
    }
    if (pl->dev) pool_free(pl->dev);
    if (pl->ts) pool_free(pl->ts);
    delete pl;
    return st;
}

}  // extern "C"
