// The layer push on the host side: the library's device memory pool, status stream, push lanes and
// event pool, the plan upload, the side-stream issue path, completion counting, per-layer status and
// the read-back of the kernels' timing stamps. The copy kernels themselves are in kvx_copy.cu.
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
    pl->off_runs = pl->off_err + align_up(sizeof(int32_t) * (size_t)pl->src.n_layers, a);
    pl->off_maps = pl->off_runs + align_up(sizeof(int32_t) * 3 * (size_t)pl->run_cap, a);
    pl->dev_bytes = pl->off_maps + align_up(sizeof(CUtensorMap) * pl->maps.size(), a);
}

// ------------------------------------------------------------------------------------------------
// Tensor maps (TENSOR plans)
// ------------------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Maps already encoded, by (buffer base, side geometry, box, box order): plans rebuilt every step over
// the same pools find theirs here instead of encoding one per buffer again.
using MapKey = std::tuple<uintptr_t, int32_t, int32_t, int32_t, int64_t, int64_t, int32_t, int32_t, int32_t>;
static std::mutex g_map_mu;
static std::map<MapKey, CUtensorMap> g_map_cache;

// One side's buffer as a rank-4 tensor of 8-byte elements. In box order NHD the dimensions are
// (head bytes / 8, head, token slot, block), in box order HND (head bytes / 8, token slot, head,
// block); the strides come from the side's own layout (NHD: a head's row follows the previous head's,
// a slot follows all heads; HND: a slot's row follows the previous slot's, a head follows all slots).
// The box is (head bytes / 8, box_k heads, box_n slots, 1 block) in the order's dimensions, so a load
// lands in shared memory in the box order whichever the side's layout, and a store writes the box
// back in the side's layout.
static bool encode_one(const Geom &g, void *base, int32_t box_n, int32_t box_k, int32_t order, CUtensorMap *out) {
    const MapKey key{(uintptr_t)base, g.layout, g.block_size, g.heads_per_shard, g.head_bytes(), g.n_blocks, box_n,
                     box_k, order};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_map_cache.find(key);
        if (it != g_map_cache.end()) { *out = it->second; return true; }
    }
    EncodeTiledFn enc = encoder();
    if (!enc || g.n_blocks < 1) return false;
    const int64_t hb = g.head_bytes();
    const cuuint64_t row = (cuuint64_t)g.row_bytes(), blk = (cuuint64_t)g.block_size * row;
    // byte strides of one head and one slot in the side's layout
    const cuuint64_t head_stride = g.layout == KVX_LAYOUT_HND ? (cuuint64_t)(g.block_size * hb) : (cuuint64_t)hb;
    const cuuint64_t slot_stride = g.layout == KVX_LAYOUT_HND ? (cuuint64_t)hb : row;
    const bool hnd = order == KVX_LAYOUT_HND;
    const cuuint64_t dim[4] = {(cuuint64_t)(hb / 8), hnd ? (cuuint64_t)g.block_size : (cuuint64_t)g.heads_per_shard,
                               hnd ? (cuuint64_t)g.heads_per_shard : (cuuint64_t)g.block_size, (cuuint64_t)g.n_blocks};
    const cuuint64_t stride[3] = {hnd ? slot_stride : head_stride, hnd ? head_stride : slot_stride, blk};
    const cuuint32_t box[4] = {(cuuint32_t)(hb / 8), (cuuint32_t)(hnd ? box_n : box_k), (cuuint32_t)(hnd ? box_k : box_n),
                               1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    const CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, base, dim, stride, box, elem,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_cache.size() >= 65536) g_map_cache.clear();
    g_map_cache.emplace(key, *out);
    return true;
}

bool encode_tensor_maps(kvx_plan_s *pl) {
    const size_t ns = pl->src_base.size(), nd = pl->dst_base.size();
    pl->maps.resize(ns + nd);
    for (size_t i = 0; i < ns; ++i)
        if (!encode_one(pl->src, pl->src_base[i], pl->box_n, pl->box_k, pl->box_order, &pl->maps[i])) {
            pl->maps.clear();
            return false;
        }
    for (size_t i = 0; i < nd; ++i)
        if (!encode_one(pl->dst, pl->dst_base[i], pl->box_n, pl->box_k, pl->box_order, &pl->maps[ns + i])) {
            pl->maps.clear();
            return false;
        }
    return true;
}

static int32_t log2_or_minus1(int64_t v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int32_t k = 0;
    while ((int64_t)1 << k != v) ++k;
    return k;
}

static TensorSide tensor_side(const kvx_plan_s *pl, const Geom &g) {
    TensorSide t;
    t.flat = tensor_side_flat(g, pl->box_order, pl->box_n, pl->box_k);
    t.hb = g.head_bytes();
    t.layout = g.layout;
    t.bs = g.block_size;
    t.hps = g.heads_per_shard;
    t.sh_hb = log2_or_minus1(t.hb);
    t.sh_bs = log2_or_minus1(t.bs);
    t.sh_hps = log2_or_minus1(t.hps);
    return t;
}

kvx_status check_pool_memory(kvx_plan_s *pl) {
    if (pl->outside_device >= 0) return KVX_OK;
    const void *probe[4] = {pl->src_base.front(), pl->src_base.back(), pl->dst_base.front(), pl->dst_base.back()};
    int32_t outside = 0;
    for (const void *p : probe) {
        cudaPointerAttributes a;
        cudaError_t e = cudaPointerGetAttributes(&a, p);
        if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(pool buffer)");
        if (a.type == cudaMemoryTypeDevice) continue;
        outside = 1;
        if (a.type == cudaMemoryTypeUnregistered) {
            int dev = 0, pageable = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(pageable memory access)");
            if (!pageable) return fail(KVX_EINVAL, "a pool buffer is pageable host memory this GPU cannot access");
        }
    }
    pl->outside_device = outside;
    return KVX_OK;
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
    a.wait_ns = kBulkWaitNs;
    a.stall_layer = -1;
    const CUtensorMap *maps =
        pl->maps.empty() ? nullptr : reinterpret_cast<const CUtensorMap *>(base + pl->off_maps);
    a.src_maps = maps;
    a.dst_maps = maps ? maps + pl->src_base.size() : nullptr;
    a.ts = tensor_side(pl, pl->src);
    a.td = tensor_side(pl, pl->dst);
    a.box_n = pl->box_n;
    a.box_k = pl->box_k;
    a.box_order = pl->box_order;
    a.n_tiles = pl->n_tiles;
    a.src_buf_bytes = pl->src.buf_bytes();
    a.dst_buf_bytes = pl->dst.buf_bytes();
    a.src_pitch = pl->src_pitch;
    a.dst_pitch = pl->dst_pitch;
    a.src_head_pitch = pl->src_head_pitch;
    a.dst_head_pitch = pl->dst_head_pitch;
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
    kvx_status st = check_pool_memory(pl);
    if (st) return st;
    // TENSOR plans encode a tensor map per buffer; a map the driver refuses sends the plan to PERSIST
    if (effective_kernel(pl) == KVX_KERNEL_TENSOR && !encode_tensor_maps(pl)) pl->kernel = KVX_KERNEL_PERSIST;
    plan_layout(pl);
    st = pool_alloc(&pl->dev, pl->dev_bytes, stream);
    if (st) return st;
    // one host image of the descriptor block, uploaded with a single copy; the plan keeps the image
    // until it is destroyed, so the copy never reads freed host memory
    pl->upload_img.assign(pl->dev_bytes, 0);
    uint8_t *img = pl->upload_img.data();
    if (pl->n_tiles) memcpy(img + pl->off_tiles, pl->tiles.data(), sizeof(TileDesc) * (size_t)pl->n_tiles);
    memcpy(img + pl->off_src, pl->src_base.data(), sizeof(void *) * pl->src_base.size());
    memcpy(img + pl->off_dst, pl->dst_base.data(), sizeof(void *) * pl->dst_base.size());
    if (!pl->maps.empty()) memcpy(img + pl->off_maps, pl->maps.data(), sizeof(CUtensorMap) * pl->maps.size());
    cudaError_t e = cudaMemcpyAsync(pl->dev, img, pl->dev_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(plan upload)");
    st = event_take(&pl->upload_evt);
    if (st) return st;
    e = cudaEventRecord(pl->upload_evt, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(upload)");
    pl->upload_stream = stream;
    e = cudaGetDevice(&pl->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
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

// Layers one launch of a push over `n` layers covers: the plan's request, else with lanes a count
// that moves about kLaunchTargetBytes per launch (long single launches of many layers ran slower on
// GB300 than launches of a few hundred MiB overlapping on the lanes), else all of them.
static int32_t layers_per_launch(const kvx_plan_s *pl, int32_t n) {
    if (pl->layers_per_launch_req > 0) return std::min(n, pl->layers_per_launch_req);
    if (pl->lanes <= 1) return n;
    const int64_t per_layer = std::max<int64_t>(1, 2 * pl->bytes_per_layer);
    return (int32_t)std::min<int64_t>(n, std::max<int64_t>(1, kLaunchTargetBytes / per_layer));
}

// Lanes at `stream`'s priority, looked up once per caller stream.
static kvx_status lanes_for(kvx_plan_s *pl, cudaStream_t stream) {
    if (pl->lane_src == stream && (int32_t)pl->lane_cache.size() == pl->lanes) return KVX_OK;
    int prio = 0;
    cudaError_t e = cudaStreamGetPriority(stream, &prio);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetPriority");
    pl->lane_cache.assign(pl->lanes, nullptr);
    for (int32_t i = 0; i < pl->lanes; ++i) {
        kvx_status st = lane_stream(i, prio, &pl->lane_cache[i]);
        if (st) return st;
    }
    pl->lane_src = stream;
    return KVX_OK;
}

// One copy launch for layers [l0, l1) on `stream`, tracked as a pending push.
static kvx_status launch_tracked(kvx_plan_s *pl, int32_t l0, int32_t l1, cudaStream_t stream, cudaEvent_t *ev_out) {
    int32_t slot = -1;
    if ((pl->flags & KVX_PLAN_TIMING) && (int32_t)pl->pending.size() < kTimingSlots) slot = (int32_t)pl->pending.size();
    const LaunchShape shape{effective_kernel(pl), pl->vec, pl->strided, pl->threads, pl->tile_bytes, pl->ctas_per_sm,
                            pl->bulk_stages, pl->per_head, pl->max_ctas};
    CopyArgs args = plan_copy_args(pl, l0);
    if (slot >= 0) {
        args.ts_start = pl->ts + slot;
        args.ts_end = pl->ts + kTimingSlots + slot;
    }
    for (int32_t l = l0; l < l1 && (ring_kernel(shape.kernel) || staged_kernel(shape.kernel)); ++l) {
        if (!pl->stall[l]) continue;
        args.stall_layer = l;              // testing hook: one stage of this layer never completes
        args.wait_ns = kBulkStallWaitNs;
        pl->stall[l] = 0;
        break;
    }
    // the completion event is taken before the launch, so a launched push is always tracked
    cudaEvent_t ev;
    kvx_status st = take_event(pl, &ev);
    if (st) return st;
    cudaError_t e = launch_copy(args, l1 - l0, shape, stream);
    if (e != cudaSuccess) {
        pl->free_events.push_back(ev);
        for (int32_t l = l0; l < l1; ++l) pl->layer_state[l] = KVX_LAYER_FAILED;
        return cuda_fail(e, "copy kernel launch");
    }
    e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) {
        // launched but not trackable: the layers cannot be confirmed
        pl->free_events.push_back(ev);
        for (int32_t l = l0; l < l1; ++l) pl->layer_state[l] = KVX_LAYER_FAILED;
        return cuda_fail(e, "cudaEventRecord(push)");
    }
    pl->pending.push_back({ev, slot, l0, l1});
    for (int32_t l = l0; l < l1; ++l) {
        pl->layer_state[l] = KVX_LAYER_PENDING;
        if (pl->inject[l]) { pl->injected_pending[l] = 1; pl->inject[l] = 0; }
    }
    *ev_out = ev;
    return KVX_OK;
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
    // timing plans: stamps live in a buffer set up on the caller's stream before the fork, so every
    // lane sees it initialised
    if (pl->flags & KVX_PLAN_TIMING) {
        st = ensure_timing_slots(pl, stream);
        if (st) return st;
    }
    if (pl->lanes > 1) {
        // fork: each lane used below waits for everything already on the caller's stream (the
        // upload included)
        if (!pl->fork_evt) {
            st = event_take(&pl->fork_evt);
            if (st) return st;
        }
        e = cudaEventRecord(pl->fork_evt, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
        st = lanes_for(pl, stream);
        if (st) return st;
    }
    const int32_t per = layers_per_launch(pl, l1 - l0);
    cudaStream_t last = stream;
    int32_t last_lane = -1;
    cudaEvent_t lane_last[8] = {};   // this call's latest launch on each lane (lanes <= 8)
    for (int32_t c0 = l0; c0 < l1; c0 += per) {
        const int32_t c1 = std::min(l1, c0 + per);
        cudaStream_t run = stream;
        int32_t li = -1;
        if (pl->lanes > 1) {
            li = pl->next_lane;
            run = pl->lane_cache[li];
            pl->next_lane = (pl->next_lane + 1) % pl->lanes;
            e = cudaStreamWaitEvent(run, pl->fork_evt, 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(fork)");
        }
        if (ready) {
            e = cudaStreamWaitEvent(run, ready, 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(ready)");
        }
        cudaEvent_t ev = nullptr;
        st = launch_tracked(pl, c0, c1, run, &ev);
        if (st) return st;
        if (li >= 0) lane_last[li] = ev;
        last = run;
        last_lane = li;
    }
    if (done) {
        // `done` follows every launch of the call: the last launch's stream joins the other lanes
        for (int32_t i = 0; i < 8; ++i) {
            if (!lane_last[i] || i == last_lane) continue;
            e = cudaStreamWaitEvent(last, lane_last[i], 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(join)");
        }
        e = cudaEventRecord(done, last);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(done)");
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
    const DeviceScope on_device(pl->device);   // read-backs, the event pool and frees of the plan's device
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
    const DeviceScope on_device(pl->device);   // read-backs, the event pool and frees of the plan's device
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
