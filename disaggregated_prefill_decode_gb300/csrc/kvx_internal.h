// Internal definitions shared by the kvx translation units (not installed; the public ABI is kvx.h).
#pragma once

#include "kvx.h"

#include <cuda.h>   // CUtensorMap (the type; the encoder is fetched from the driver at run time)

#include <atomic>
#include <cstdint>
#include <vector>

namespace kvx {

// One tile of copy work: a CTA moves it for one (layer, plane). Offsets are bytes into the
// producer / consumer buffer of (layer, plane, shard). Contiguous plans: `n` is a byte count.
// Strided plans (head-shard remap): `n` rows of CopyArgs::width bytes at the two row pitches, for
// each of `heads` heads (0 and 1 both mean one) at the two head pitches: row t of head h is at
// off + h * head_pitch + t * pitch on each side.
struct alignas(16) TileDesc {
    int64_t src_off;
    int64_t dst_off;
    int32_t n;
    int32_t s_shard;
    int32_t d_shard;
    int32_t heads;
};
static_assert(sizeof(TileDesc) == 32, "TileDesc is two 16-byte words");

// TENSOR plans: what the kernel needs to turn a tile's byte offsets into tensor-map coordinates
// (head, slot, block) on each side, and the maps' box (box_n token slots x box_k heads, laid out in
// shared memory in the plan's box order: KVX_LAYOUT_NHD slot-major, KVX_LAYOUT_HND head-major).
struct TensorSide {
    int64_t hb;                       // head bytes
    int32_t layout, bs, hps;
    int32_t sh_hb, sh_bs, sh_hps;     // log2 of hb / bs / hps when a power of two, else -1
    int32_t flat;                     // a box is one contiguous span on this side, in the box order:
                                      // moved by one plain bulk copy instead of a tensor-map copy
};

// Kernel arguments of one push launch (passed by value).
struct CopyArgs {
    const TileDesc *tiles;
    const uint8_t *const *src_base;   // [n_layers][n_planes][src_shards] device pointers
    uint8_t *const *dst_base;         // [n_layers][n_planes][dst_shards]
    int32_t *err;                     // [n_layers] error words, set only when a tile is out of bounds
    int64_t n_tiles;                  // tiles per (layer, plane)
    int64_t src_buf_bytes;
    int64_t dst_buf_bytes;
    int64_t src_pitch;                // producer row bytes
    int64_t dst_pitch;                // consumer row bytes
    int64_t src_head_pitch;           // strided tiles of several heads: bytes from one head to the next
    int64_t dst_head_pitch;
    unsigned long long *ts_start;     // timing: atomicMin of %globaltimer at each CTA's start (or null)
    unsigned long long *ts_end;       // timing: atomicMax of %globaltimer at each CTA's end
    uint64_t wait_ns;                 // bulk: limit of one wait for a ring stage (kBulkWaitNs)
    int32_t stall_layer;              // bulk, testing hook: this layer's first item on CTA 0 never completes (-1: none)
    const CUtensorMap *src_maps;      // TENSOR: one map per producer buffer (device, 64-byte aligned)
    const CUtensorMap *dst_maps;      // TENSOR: one map per consumer buffer
    TensorSide ts, td;                // TENSOR: producer / consumer geometry
    int32_t box_n, box_k;             // TENSOR: the maps' box
    int32_t box_order;                // TENSOR: KVX_LAYOUT_NHD or KVX_LAYOUT_HND (the box in shared memory)
    int32_t width;                    // strided: bytes copied per row
    int32_t n_planes;
    int32_t src_shards;
    int32_t dst_shards;
    int32_t layer0;
};

struct Geom {
    int32_t n_layers, n_planes, n_shards, heads_per_shard, head_dim, elem_bytes, block_size;
    int32_t layout;                   // KVX_LAYOUT_NHD or KVX_LAYOUT_HND
    int64_t n_blocks;
    // index of (block, slot, head) inside one buffer, in units of head_bytes()
    int64_t head_index(int64_t blk, int64_t slot, int64_t head) const {
        return layout == KVX_LAYOUT_HND ? (blk * heads_per_shard + head) * block_size + slot
                                        : (blk * block_size + slot) * heads_per_shard + head;
    }
    // bytes between consecutive tokens of one head inside a block
    int64_t token_pitch() const { return layout == KVX_LAYOUT_HND ? head_bytes() : row_bytes(); }
    int64_t head_bytes() const { return (int64_t)head_dim * elem_bytes; }
    int64_t row_bytes() const { return (int64_t)heads_per_shard * head_bytes(); }
    int64_t buf_bytes() const { return n_blocks * block_size * row_bytes(); }
    int32_t n_buffers() const { return n_layers * n_planes * n_shards; }
};

// Makes `device` current for a scope and restores the caller's device after it; nothing happens
// for -1 or when that device is already current.
struct DeviceScope {
    int prev = -1;
    explicit DeviceScope(int device) {
        if (device < 0 || cudaGetDevice(&prev) != cudaSuccess || prev == device || cudaSetDevice(device) != cudaSuccess)
            prev = -1;
    }
    ~DeviceScope() {
        if (prev >= 0) cudaSetDevice(prev);
    }
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;
};

struct PendingPush {
    cudaEvent_t done;
    int32_t slot;           // timing plans: index of its global-timer stamps, -1 when not timed
    int32_t layer_begin, layer_end;
};

// Bulk kernel: limit of one wait for a ring stage, far beyond any legitimate tile copy; and the
// limit a push armed by kvx_plan_inject_stall runs with.
constexpr uint64_t kBulkWaitNs = 2000000000ull;        // 2 s
constexpr uint64_t kBulkStallWaitNs = 1000000ull;      // 1 ms

// Timing plans: pushes between two syncs that can carry global-timer stamps.
constexpr int32_t kTimingSlots = 4096;

// Bytes moved (read + write) one launch of a multi-layer push aims at when it is split over lanes.
constexpr int64_t kLaunchTargetBytes = (int64_t)256 << 20;

// Bulk copy launches that read at least this many bytes mark what they touch evict-first in L2.
constexpr int64_t kStreamL2Bytes = (int64_t)8 << 20;

// Head-shard pair: the contiguous head range one producer shard shares with one consumer shard, as
// byte offsets inside a producer row and a consumer row.
struct Pair { int32_t s, d; int64_t src_seg_off, dst_seg_off; };
std::vector<Pair> shard_pairs(const Geom &s, const Geom &d);

// Thread-local error text; returns `st` so call sites can `return fail(st, ...)`.
kvx_status fail(kvx_status st, const char *fmt, ...);
kvx_status cuda_fail(cudaError_t e, const char *what);
void count_launch(int64_t n = 1);
size_t align_up(size_t x, size_t a);

// Device memory from a library-owned stream-ordered pool (one per device; it keeps freed memory
// for reuse instead of returning it to the driver at every synchronisation).
kvx_status pool_alloc(void **ptr, size_t bytes, cudaStream_t stream);
void pool_free(void *ptr);
// A non-blocking stream per device for the library's own small read-backs.
kvx_status aux_stream(cudaStream_t *out);
// Library-wide pool of events per (device, timing): plans rebuilt every step reuse them instead of
// creating and destroying one or two per push.
kvx_status event_take(cudaEvent_t *ev);
void event_give(cudaEvent_t ev);

// Launches the tile copy for layers [args.layer0, args.layer0 + n_layers) (kvx_push.cu).
struct LaunchShape {
    int32_t kernel;        // KVX_KERNEL_TILE / PERSIST / BULK (resolved)
    int32_t vec;
    int32_t strided;
    int32_t threads;
    int32_t tile_bytes;    // bulk: bytes per stage
    int32_t ctas_per_sm;   // 0: occupancy limit
    int32_t stages;        // bulk: ring stages (2, 3, 4, 6 or 8)
    int32_t head_groups;   // tiles are head groups (a head-major side): many small row copies per tile
    int32_t max_ctas;      // upper bound on the launch's CTAs (0: none)
};
cudaError_t launch_copy(const CopyArgs &args, int32_t n_layers, const LaunchShape &shape, cudaStream_t stream);

// Bulk ring: stage counts with a kernel instantiation, and the most shared memory one ring may take
// (two rings of an overlapping push then still fit an SM's 228 KiB only when each is <= 113 KiB).
constexpr int64_t kBulkRingMax = 192 << 10;
inline bool valid_stages(int32_t s) { return s == 0 || s == 2 || s == 3 || s == 4 || s == 6 || s == 8; }

}  // namespace kvx

// The plan object behind kvx_plan_t.
struct kvx_plan_s {
    kvx::Geom src{}, dst{};
    std::vector<void *> src_base, dst_base;   // host copies of the pools' pointer tables

    // merged token runs (host), rows = block * block_size + slot
    std::vector<int32_t> run_src_row, run_dst_row, run_ntok;

    // copy shape
    int32_t strided = 0;
    int32_t per_head = 0;                      // tiles are (block segment, head) pieces (an HND side)
    int64_t src_pitch = 0, dst_pitch = 0;      // strided tiles: row pitches
    int64_t src_head_pitch = 0, dst_head_pitch = 0;   // per-head plans: head pitches of head-group tiles
    int32_t vec = 16;
    int32_t width = 0;
    int32_t tile_bytes = 16384;
    int32_t threads = 256;                     // resolved threads per CTA of TILE / PERSIST
    int32_t threads_req = 0;                   // threads asked for (0: by plan size)
    int32_t flags = 0;                         // KVX_PLAN_* bits
    int32_t kernel = 0;                        // resolved KVX_KERNEL_*
    int32_t ctas_per_sm = 0;                   // resident CTAs per SM of persistent kernels (0: by size)
    int32_t lanes = 4;                         // internal streams pushes fan out over (default_lanes())
    int32_t bulk_stages_req = 0;               // ring stages asked for (0: by plan kind)
    int32_t bulk_stages = 4;                   // ring stages of the bulk kernel, resolved
    int32_t layers_per_launch_req = 0;         // kvx_push_layers: layers per launch asked for (0: by size)
    int32_t max_ctas = 0;                      // upper bound on CTAs per copy launch (0: none)
    int32_t box_n = 0, box_k = 0;              // TENSOR: token slots x heads of a tile the maps move at once
    int32_t box_order = KVX_LAYOUT_NHD;        // TENSOR: layout of the box in shared memory
    bool head_tile_auto = false;               // head-group tiles of the library's default size
    std::vector<CUtensorMap> maps;             // TENSOR: producer buffers' maps, then consumer buffers' (host)
    int32_t outside_device = -1;               // a pool buffer outside device memory (-1: not checked yet)
    int32_t next_lane = 0;
    cudaEvent_t fork_evt = nullptr;            // recorded on the caller's stream before each lane push
    cudaStream_t lane_src = nullptr;           // caller stream the cached lanes below were chosen for
    std::vector<cudaStream_t> lane_cache;      // lanes at that stream's priority
    int64_t n_tiles = 0;                       // per (layer, plane)
    int64_t bytes_per_layer = 0;
    std::vector<kvx::TileDesc> tiles;          // host-built plans; empty for device-built plans

    // device copy: [tiles][src_base][dst_base][err][runs: device-built plans only]
    void *dev = nullptr;
    size_t dev_bytes = 0;
    size_t off_tiles = 0, off_src = 0, off_dst = 0, off_err = 0, off_runs = 0, off_maps = 0;
    int64_t run_cap = 0;                       // device-built plans: run slots (src rows, dst rows, tokens)
    int64_t n_runs_dev = -1;                   // device-built plans: runs held on the device until asked for
    int64_t device_tokens = 0;                 // device-built plans: tokens copied per (layer, plane, shard)
    std::vector<uint8_t> upload_img;           // host image of the uploaded descriptor bytes
    bool uploaded = false;
    int32_t device = -1;                       // device of the descriptors, set when they are uploaded
    bool device_built = false;                 // descriptors were written on the device
    cudaEvent_t upload_evt = nullptr;
    cudaStream_t upload_stream = nullptr;

    // pushes issued and not yet confirmed by kvx_sync
    std::vector<kvx::PendingPush> pending;
    std::vector<cudaEvent_t> free_events;
    std::vector<float> push_start_us, push_end_us;   // timing plans: confirmed by the last sync
    std::vector<int64_t> push_start_ns, push_end_ns; // the same, raw device global-timer values
    unsigned long long *ts = nullptr;                // timing stamps: [kTimingSlots] starts, then ends
    std::vector<int32_t> layer_state;          // kvx_layer_state per layer
    std::vector<uint8_t> inject;               // host fault injection armed, per layer
    std::vector<uint8_t> injected_pending;     // injected failure waiting for sync, per layer
    std::vector<uint8_t> stall;                // kvx_plan_inject_stall armed, per layer
};

namespace kvx {
// The kernel a plan's pushes run: pools outside device memory (host memory over the chip-to-chip
// link, managed memory) are copied with plain loads and stores, never by the bulk copy path.
// TENSOR plans whose descriptors went up without tensor maps (the driver refused one, or the kernel
// was chosen by kvx_plan_set_opts after the first push) run PERSIST.
inline int32_t effective_kernel(const kvx_plan_s *pl) {
    const bool async_copy = pl->kernel == KVX_KERNEL_BULK || pl->kernel == KVX_KERNEL_TENSOR ||
                            pl->kernel == KVX_KERNEL_STAGED;
    if (async_copy && pl->outside_device == 1) return KVX_KERNEL_PERSIST;
    if (pl->kernel == KVX_KERNEL_TENSOR && pl->uploaded && pl->maps.empty()) return KVX_KERNEL_PERSIST;
    return pl->kernel;
}
// The ring kernels (BULK, TENSOR) run one issuing thread per 32-thread CTA; STAGED has the same
// ring with 128 threads storing.
inline bool ring_kernel(int32_t k) { return k == KVX_KERNEL_BULK || k == KVX_KERNEL_TENSOR; }
inline bool staged_kernel(int32_t k) { return k == KVX_KERNEL_STAGED; }
// Lanes of a plan that asks for none: 4, or half the process's hardware work queues
// (CUDA_DEVICE_MAX_CONNECTIONS) when that is fewer, at least 1 (kvx_plan.cpp).
int32_t default_lanes();
// TENSOR plans: encodes one tensor map per pool buffer into pl->maps (host); false when the driver
// refuses a map (the plan then runs PERSIST) (kvx_push.cu).
bool encode_tensor_maps(kvx_plan_s *pl);
// TENSOR plans: whether a box (box_n slots x box_k heads, laid out in `order`) is one contiguous span
// of a side with geometry g (kvx_tiles.cpp).
bool tensor_side_flat(const Geom &g, int32_t order, int32_t box_n, int32_t box_k);
// Checks where the pools' buffers live (first and last buffer of each side) and records it; refuses
// pageable host memory the GPU cannot reach (kvx_push.cu).
kvx_status check_pool_memory(kvx_plan_s *pl);
// Shared by host-built and device-built plans: validation (kvx_plan.cpp) and the copy shape
// (kvx_tiles.cpp).
kvx_status init_plan_geometry(const kvx_pool *src, const kvx_pool *dst, const kvx_plan_opts *opts, kvx_plan_s *pl);
void init_copy_shape(kvx_plan_s *pl, bool tile_bytes_given);
void request_runs(int64_t n_tok, int32_t bs_s, const int32_t *sids, int32_t bs_d, const int32_t *dids, kvx_plan_s *pl);
void build_tiles(kvx_plan_s *pl);
void finish_plan_shape(kvx_plan_s *pl);
void resolve_launch(kvx_plan_s *pl);        // kernel, threads and ring stages from the plan's options
bool as_whole_block_copy(kvx_plan_s *pl);
// Device layout and kernel arguments of a plan (kvx_push.cu).
void plan_layout(kvx_plan_s *pl);
CopyArgs plan_copy_args(const kvx_plan_s *pl, int32_t layer0);
}  // namespace kvx
