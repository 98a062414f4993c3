// The copy kernels of the layer push for sm_103a and their launcher: TILE (one CTA per tile),
// PERSIST (a resident grid walking the tiles) and BULK (cp.async.bulk through a shared-memory ring of
// mbarrier-tracked stages), all driven by the plan's tile table, all checking every tile against the
// buffer extents (an out-of-bounds tile sets its layer's error word instead of faulting), and all
// stamping the GPU's global timer for timing plans.
//
// Follows the push-mode NIXL connector article (spke.com 3844), "Implementierungsdetails" step 3
// (the producer writes the KV blocks straight into the consumer's memory, each side addressing its
// own layout) and the "vLLM MoRIIO KV Connector" notes, section 6 (transfers as (source offset,
// destination offset, size) with adjacent blocks merged).
#include "kvx_internal.h"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

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
    const int64_t k = STRIDED ? (int64_t)max(t.heads, 1) - 1 : 0;     // heads after the first
    const int64_t src_end =
        STRIDED ? t.src_off + (int64_t)(t.n - 1) * a.src_pitch + k * a.src_head_pitch + a.width : t.src_off + t.n;
    const int64_t dst_end =
        STRIDED ? t.dst_off + (int64_t)(t.n - 1) * a.dst_pitch + k * a.dst_head_pitch + a.width : t.dst_off + t.n;
    return t.n > 0 && t.heads >= 0 && t.src_off >= 0 && t.dst_off >= 0 && src_end <= a.src_buf_bytes &&
           dst_end <= a.dst_buf_bytes && t.s_shard >= 0 && t.s_shard < a.src_shards && t.d_shard >= 0 &&
           t.d_shard < a.dst_shards;
}

// Rows of a strided tile in head-major order: row r is row r % n of head r / n. A thread walks its
// rows r0, r0 + step, ... keeping (head, row) by subtraction instead of dividing for every row.
struct RowCursor {
    int32_t h, t, n;
    __device__ __forceinline__ RowCursor(int32_t r0, int32_t n_) : h(r0 / n_), t(r0 - (r0 / n_) * n_), n(n_) {}
    __device__ __forceinline__ void advance(int32_t step) {
        t += step;
        while (t >= n) { t -= n; ++h; }
    }
};

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
        // Rows of `width` bytes at the two pitches, for each of the tile's heads. Threads are laid
        // out as (row lane, column) once, so the loop has no per-element division.
        const int32_t vpr = a.width / VEC;
        const int32_t rows = t.n * max(t.heads, 1);
        if (vpr <= (int32_t)blockDim.x) {
            const int32_t rpp = (int32_t)blockDim.x / vpr;          // rows per pass
            const int32_t my_row = (int32_t)threadIdx.x / vpr;
            const int32_t col = (int32_t)threadIdx.x - my_row * vpr;
            if (my_row < rpp) {
                RowCursor c(my_row, t.n);
                for (int32_t row = my_row; row < rows; row += rpp * kUnroll) {
                    V r[kUnroll];
                    int64_t so[kUnroll], dof[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        so[u] = (int64_t)c.h * a.src_head_pitch + (int64_t)c.t * a.src_pitch;
                        dof[u] = (int64_t)c.h * a.dst_head_pitch + (int64_t)c.t * a.dst_pitch;
                        c.advance(rpp);
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        if (row + u * rpp < rows) r[u] = reinterpret_cast<const V *>(src + so[u])[col];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        if (row + u * rpp < rows) reinterpret_cast<V *>(dst + dof[u])[col] = r[u];
                }
            }
        } else {
            for (int32_t row = 0; row < rows; ++row) {
                const int32_t h = row / t.n, tr = row - h * t.n;
                const V *s = reinterpret_cast<const V *>(src + (int64_t)h * a.src_head_pitch + (int64_t)tr * a.src_pitch);
                V *d = reinterpret_cast<V *>(dst + (int64_t)h * a.dst_head_pitch + (int64_t)tr * a.dst_pitch);
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
// A strided tile (rows of `width` bytes at each side's pitch, for each head of a head group) is packed
// densely in its stage, head-major or token-major: a side whose rows lie adjacent in that order moves
// in one bulk copy, the other piece by piece, all pieces of a load completing on the stage's one
// mbarrier and all stores of a stage forming one bulk group.
// ------------------------------------------------------------------------------------------------

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

// Bounded wait for a stage's phase; false when `limit_ns` passed. Each try_wait already suspends
// the thread for a while when the phase is not complete; the global timer (a costly special register
// to read, and issue slots taken from the SM's other warps) is read only every 64 tries.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t k = 1;; ++k) {
        if (mbar_test(bar, parity)) return true;
        if ((k & 63) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// An L2 access policy that marks the lines a copy touches evict-first. A contiguous launch that
// streams many MiB through L2 passes it with its loads and its stores: on GB300 the per-layer push
// step of a 8192-token request then ran at 0.983-0.990 of the copy peak against 0.961-0.969 without
// (loads alone 0.939, stores alone 0.964).
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_load(void *stage, const void *src, uint32_t bytes, uint64_t *bar, bool hint,
                                          uint64_t policy) {
    if (hint)
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
                     "[%3], %4;" ::"r"(smem_addr(stage)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
                     : "memory");
    else
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_addr(stage)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                     : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *stage, uint32_t bytes, bool hint, uint64_t policy) {
    if (hint)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                     "r"(smem_addr(stage)), "r"(bytes), "l"(policy)
                     : "memory");
    else
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
    int32_t n;         // strided tiles: rows of a.width bytes per head; contiguous tiles: 1
    int32_t heads;     // strided tiles: heads of the group (1 for a single head)
    int32_t layer;
    int32_t tensor;    // TENSOR: the tile is the maps' box: one copy each way (a plain bulk copy on a
                       // side that holds the box as one span, else a tensor-map copy)
    int32_t s_buf, d_buf;             // TENSOR: buffer (map) index on each side
    int32_t sh, ss, sb, dh, ds, db;   // TENSOR: (head, slot, block) of the tile on each side
};

__device__ __forceinline__ int64_t div_by(int64_t x, int64_t d, int32_t shift) { return shift >= 0 ? x >> shift : x / d; }

// (block, slot, head) of a byte offset into one side's buffer: the offset is head_index * head bytes,
// head_index = (block * bs + slot) * hps + head (NHD) or (block * hps + head) * bs + slot (HND).
__device__ __forceinline__ void side_coords(const TensorSide &g, int64_t off, int32_t *blk, int32_t *slot, int32_t *head) {
    const int64_t idx = div_by(off, g.hb, g.sh_hb);
    if (g.layout == KVX_LAYOUT_HND) {
        const int64_t r = div_by(idx, g.bs, g.sh_bs);
        const int64_t b = div_by(r, g.hps, g.sh_hps);
        *slot = (int32_t)(idx - r * g.bs);
        *head = (int32_t)(r - b * g.hps);
        *blk = (int32_t)b;
    } else {
        const int64_t r = div_by(idx, g.hps, g.sh_hps);
        const int64_t b = div_by(r, g.bs, g.sh_bs);
        *head = (int32_t)(idx - r * g.hps);
        *slot = (int32_t)(r - b * g.bs);
        *blk = (int32_t)b;
    }
}

template <bool STRIDED, bool TENSOR>
__device__ __forceinline__ BulkItem bulk_item(const CopyArgs &a, int64_t w, int32_t stage_bytes) {
    int64_t tile, lp;
    BulkItem it;
    decode_item(a, w, &tile, &it.layer, &lp);
    const TileDesc t = a.tiles[tile];
    it.src = nullptr;
    it.dst = nullptr;
    it.bytes = 0;
    it.tensor = 0;
    it.n = STRIDED ? t.n : 1;
    it.heads = STRIDED ? max(t.heads, 1) : 1;
    const int64_t bytes = STRIDED ? (int64_t)t.n * it.heads * a.width : (int64_t)t.n;
    if (!tile_in_bounds<STRIDED>(t, a) || bytes > stage_bytes) {
        if (t.n != 0) atomicOr(&a.err[it.layer], 1);
        return it;
    }
    it.src = a.src_base[lp * a.src_shards + t.s_shard] + t.src_off;
    it.dst = a.dst_base[lp * a.dst_shards + t.d_shard] + t.dst_off;
    uintptr_t mis = ((uintptr_t)it.src) | ((uintptr_t)it.dst) | (uintptr_t)bytes;
    if (STRIDED)
        mis |= (uintptr_t)a.width | (uintptr_t)a.src_pitch | (uintptr_t)a.dst_pitch |
               (it.heads > 1 ? (uintptr_t)(a.src_head_pitch | a.dst_head_pitch) : 0);
    if (mis & 15) {
        atomicOr(&a.err[it.layer], 1);
        return it;
    }
    it.bytes = (uint32_t)bytes;
    if (TENSOR && t.n == a.box_n && it.heads == a.box_k) {
        // the maps' box: one copy each way when it stays inside a block and a shard on both sides
        side_coords(a.ts, t.src_off, &it.sb, &it.ss, &it.sh);
        side_coords(a.td, t.dst_off, &it.db, &it.ds, &it.dh);
        it.s_buf = (int32_t)(lp * a.src_shards + t.s_shard);
        it.d_buf = (int32_t)(lp * a.dst_shards + t.d_shard);
        it.tensor = it.ss + a.box_n <= a.ts.bs && it.sh + a.box_k <= a.ts.hps && it.ds + a.box_n <= a.td.bs &&
                    it.dh + a.box_k <= a.td.hps;
    }
    return it;
}

// Tensor-map copies of one box (rank 4: head bytes / 8, then head and slot in the plan's box order,
// block; x always 0; c1, c2 are the head and slot coordinates in that order). The load
// completes on the stage's mbarrier; the store joins the thread's current bulk group.
// With `hint` both carry the evict-first L2 policy (launches that stream 8 MiB or more: on GB300 a
// 32 MiB-per-layer head-layout push went from 0.836-0.844 to 0.873-0.874 of the copy peak in the
// per-layer step with it, 0.61-0.62 to 0.62-0.63 alone, a 497 MB layer unchanged at 0.99).
__device__ __forceinline__ void tensor_load(void *stage, const CUtensorMap *map, int32_t c1, int32_t c2, int32_t blk,
                                            uint64_t *bar, bool hint, uint64_t policy) {
    if (hint)
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
            "[%1, {%2, %3, %4, %5}], [%6], %7;"
            ::"r"(smem_addr(stage)), "l"(map), "r"(0), "r"(c1), "r"(c2), "r"(blk), "r"(smem_addr(bar)), "l"(policy)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
            ::"r"(smem_addr(stage)), "l"(map), "r"(0), "r"(c1), "r"(c2), "r"(blk), "r"(smem_addr(bar))
            : "memory");
}

__device__ __forceinline__ void tensor_store(const CUtensorMap *map, int32_t c1, int32_t c2, int32_t blk, const void *stage,
                                             bool hint, uint64_t policy) {
    if (hint)
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3, %4}], [%5], %6;"
                     ::"l"(map), "r"(0), "r"(c1), "r"(c2), "r"(blk), "r"(smem_addr(stage)), "l"(policy)
                     : "memory");
    else
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                     ::"l"(map), "r"(0), "r"(c1), "r"(c2), "r"(blk), "r"(smem_addr(stage))
                     : "memory");
}

// The maps live in global memory, written by the plan upload; a CTA acquires each map for the tensor
// proxy before its first use.
__device__ __forceinline__ void map_acquire(const CUtensorMap *map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

template <int STAGES, bool STRIDED, bool TENSOR>
__global__ void __launch_bounds__(32) kvx_copy_bulk(CopyArgs a, int64_t n_work, int32_t stage_bytes,
                                                     int32_t stream_l2) {
    constexpr int kBulkStages = STAGES;
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bar[kBulkStages];
    if (threadIdx.x != 0) return;
    stamp_start(a);
    const bool hint = stream_l2 != 0;
    const uint64_t policy = hint ? evict_first_policy() : 0ull;
    for (int s = 0; s < kBulkStages; ++s) mbar_init(&bar[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    const int64_t n_mine = (int64_t)blockIdx.x < n_work ? (n_work - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    BulkItem items[kBulkStages];
    // item i of this CTA is work item blockIdx.x + i * gridDim.x, in stage i % kBulkStages. A side
    // whose rows (and heads) are adjacent moves a tile in one bulk copy; the other row by row.
    auto packed = [&](const BulkItem &it, int64_t pitch, int64_t head_pitch) {
        return !STRIDED || (pitch == a.width && (it.heads == 1 || head_pitch == (int64_t)it.n * a.width));
    };
    // Stage order of a head group: head-major (row t of head h at h * n + t) unless the producer keeps
    // the group's heads of one token adjacent and the consumer does not; then token-major
    // (t * heads + h), so that each token's heads load in one copy and the rows go out one by one
    // (on GB300 row-by-row loads cost more than row-by-row stores).
    auto token_major = [&](const BulkItem &it) {
        return STRIDED && it.heads > 1 && a.src_head_pitch == a.width && a.dst_head_pitch != a.width;
    };
    const CUtensorMap *fenced_src = nullptr, *fenced_dst = nullptr;   // TENSOR: maps acquired so far
    auto issue = [&](int64_t i) {
        const int s = (int)(i % kBulkStages);
        const BulkItem it = bulk_item<STRIDED, TENSOR>(a, blockIdx.x + i * gridDim.x, stage_bytes);
        items[s] = it;
        mbar_arrive_expect(&bar[s], it.bytes);
        if (!it.bytes) return;
        uint8_t *stage = ring + (size_t)s * stage_bytes;
        if (TENSOR && it.tensor && !a.ts.flat) {
            const CUtensorMap *map = a.src_maps + it.s_buf;
            if (map != fenced_src) { map_acquire(map); fenced_src = map; }
            const bool hnd = a.box_order == KVX_LAYOUT_HND;
            tensor_load(stage, map, hnd ? it.ss : it.sh, hnd ? it.sh : it.ss, it.sb, &bar[s], hint, policy);
        } else if (TENSOR && it.tensor) {
            bulk_load(stage, it.src, it.bytes, &bar[s], hint, policy);   // the box is this side's span
        } else if (token_major(it)) {
            const uint32_t span = (uint32_t)(it.heads * a.width);    // one token's heads
            if (a.src_pitch == (int64_t)span) {
                bulk_load(stage, it.src, it.bytes, &bar[s], hint, policy);
            } else {
                for (int32_t r = 0; r < it.n; ++r)
                    bulk_load(stage + (size_t)r * span, it.src + (int64_t)r * a.src_pitch, span, &bar[s], hint, policy);
            }
        } else if (packed(it, a.src_pitch, a.src_head_pitch)) {
            bulk_load(stage, it.src, it.bytes, &bar[s], hint, policy);
        } else {
            for (int32_t h = 0; h < it.heads; ++h)
                for (int32_t r = 0; r < it.n; ++r)
                    bulk_load(stage + (size_t)(h * it.n + r) * a.width,
                              it.src + (int64_t)h * a.src_head_pitch + (int64_t)r * a.src_pitch, (uint32_t)a.width,
                              &bar[s], hint, policy);
        }
    };
    int64_t issued = 0;
    for (; issued < n_mine && issued < kBulkStages - 1; ++issued) issue(issued);
    bool timed_out = false;
    bool stall = a.stall_layer >= 0 && blockIdx.x == 0;   // testing hook (kvx_plan_inject_stall)
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = (int)(i % kBulkStages);
        const uint32_t parity = (uint32_t)((i / kBulkStages) & 1);
        bool landed = mbar_wait(&bar[s], parity, a.wait_ns);
        if (landed && stall && items[s].layer == a.stall_layer) {
            // the hook: after the stage's loads have landed, wait for the stage's next phase, which
            // nothing arms before this wait ends -- a wait that can only run out, with no copy in flight
            stall = false;
            landed = mbar_wait(&bar[s], parity ^ 1u, a.wait_ns);
        }
        if (!landed) {
            // this CTA stops here: every layer of the work it had left (items i .. n_mine - 1, in
            // layer order) is reported FAILED, not only the layer of the stage it waited for
            const int32_t per_layer = (int32_t)(a.n_tiles * a.n_planes);
            const int32_t l_last = a.layer0 + (int32_t)((blockIdx.x + (n_mine - 1) * gridDim.x) / per_layer);
            for (int32_t l = items[s].layer; l <= l_last; ++l) atomicOr(&a.err[l], 2);
            timed_out = true;
            break;
        }
        if (items[s].bytes) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint8_t *stage = ring + (size_t)s * stage_bytes;
            const BulkItem &it = items[s];
            if (TENSOR && it.tensor && !a.td.flat) {
                const CUtensorMap *map = a.dst_maps + it.d_buf;
                if (map != fenced_dst) { map_acquire(map); fenced_dst = map; }
                const bool hnd = a.box_order == KVX_LAYOUT_HND;
                tensor_store(map, hnd ? it.ds : it.dh, hnd ? it.dh : it.ds, it.db, stage, hint, policy);
            } else if (TENSOR && it.tensor) {
                bulk_store(it.dst, stage, it.bytes, hint, policy);
            } else if (token_major(it)) {
                for (int32_t h = 0; h < it.heads; ++h)
                    for (int32_t r = 0; r < it.n; ++r)
                        bulk_store(it.dst + (int64_t)h * a.dst_head_pitch + (int64_t)r * a.dst_pitch,
                                   stage + (size_t)(r * it.heads + h) * a.width, (uint32_t)a.width, hint, policy);
            } else if (packed(it, a.dst_pitch, a.dst_head_pitch)) {
                bulk_store(it.dst, stage, it.bytes, hint, policy);
            } else {
                for (int32_t h = 0; h < it.heads; ++h)
                    for (int32_t r = 0; r < it.n; ++r)
                        bulk_store(it.dst + (int64_t)h * a.dst_head_pitch + (int64_t)r * a.dst_pitch,
                                   stage + (size_t)(h * it.n + r) * a.width, (uint32_t)a.width, hint, policy);
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
            mbar_wait(&bar[i % kBulkStages], (uint32_t)((i / kBulkStages) & 1), a.wait_ns);
        }
    }
    bulk_wait_all();   // the stores have completed, not only read their stages
    if (a.ts_end) atomicMax(a.ts_end, (unsigned long long)global_ns());
}

// ------------------------------------------------------------------------------------------------
// KVX_KERNEL_STAGED: strided tiles loaded by the bulk copy engine into a shared-memory ring, then
// stored to the consumer by the CTA's threads in the consumer's own layout.
// A tile's load side is dense in one of two orders on the usual pools -- head-major (each head's n
// rows adjacent, heads n rows apart: a head-major producer) or token-major (each token's heads
// adjacent: a token-major producer) -- so it lands in one bulk copy (or one per token), in that order.
// The threads then write each row to its place on the consumer side with 16-byte stores: a head
// transpose costs no ring slot and no latency, since stores need no answer. Thread 0 issues the loads;
// all threads wait on the stage's mbarrier (bounded), copy it out, meet at a barrier, and thread 0
// refills the stage.
// ------------------------------------------------------------------------------------------------

constexpr int kStagedThreads = 128;

struct StageInfo {
    uint8_t *dst;      // consumer tile base
    uint32_t bytes;    // 0: nothing staged (skipped item)
    int32_t n;         // rows per head
    int32_t heads;
    int32_t order;     // 0: head-major (row h * n + t), 1: token-major (row t * heads + h)
    int32_t layer;
};

template <int STAGES>
__global__ void __launch_bounds__(kStagedThreads) kvx_copy_staged(CopyArgs a, int64_t n_work, int32_t stage_bytes) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bar[STAGES];
    __shared__ StageInfo info[STAGES];
    const int tid = threadIdx.x;
    if (tid == 0) {
        if (a.ts_start) atomicMin(a.ts_start, (unsigned long long)global_ns());
        for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t n_mine = (int64_t)blockIdx.x < n_work ? (n_work - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

    // thread 0: item i of this CTA (work item blockIdx.x + i * gridDim.x) into stage i % STAGES
    auto issue = [&](int64_t i) {
        const int s = (int)(i % STAGES);
        const BulkItem it = bulk_item<true, false>(a, blockIdx.x + i * gridDim.x, stage_bytes);
        StageInfo &si = info[s];
        si.dst = it.dst;
        si.bytes = it.bytes;
        si.n = it.n;
        si.heads = it.heads;
        si.layer = it.layer;
        si.order = 0;
        uint8_t *stage = ring + (size_t)s * stage_bytes;
        if (!it.bytes) {
            mbar_arrive_expect(&bar[s], 0);
            return;
        }
        const bool dense_hm = a.src_pitch == a.width && (it.heads == 1 || a.src_head_pitch == (int64_t)it.n * a.width);
        const bool tok_major = !dense_hm && it.heads > 1 && a.src_head_pitch == a.width;
        si.order = tok_major ? 1 : 0;
        mbar_arrive_expect(&bar[s], it.bytes);   // after si is written: the arrival releases it
        if (dense_hm) {
            bulk_load(stage, it.src, it.bytes, &bar[s], false, 0);
        } else if (tok_major) {
            const uint32_t span = (uint32_t)(it.heads * a.width);     // one token's heads
            if (a.src_pitch == (int64_t)span) {
                bulk_load(stage, it.src, it.bytes, &bar[s], false, 0);
            } else {
                for (int32_t r = 0; r < it.n; ++r)
                    bulk_load(stage + (size_t)r * span, it.src + (int64_t)r * a.src_pitch, span, &bar[s], false, 0);
            }
        } else {
            for (int32_t h = 0; h < it.heads; ++h)
                for (int32_t r = 0; r < it.n; ++r)
                    bulk_load(stage + (size_t)(h * it.n + r) * a.width,
                              it.src + (int64_t)h * a.src_head_pitch + (int64_t)r * a.src_pitch, (uint32_t)a.width,
                              &bar[s], false, 0);
        }
    };

    if (tid == 0)
        for (int64_t i = 0; i < n_mine && i < STAGES; ++i) issue(i);
    const int32_t vpr = a.width >> 4;                 // 16-byte vectors per row
    bool stall = a.stall_layer >= 0 && blockIdx.x == 0;   // testing hook (kvx_plan_inject_stall)
    bool timed_out = false;
    int64_t consumed = 0;
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = (int)(i % STAGES);
        const uint32_t parity = (uint32_t)((i / STAGES) & 1);
        bool landed = mbar_wait(&bar[s], parity, a.wait_ns);
        const StageInfo si = info[s];
        if (landed && stall && si.layer == a.stall_layer) {
            // the hook: once the stage's loads landed, wait for its next phase, which nothing arms
            stall = false;
            landed = mbar_wait(&bar[s], parity ^ 1u, a.wait_ns);
        }
        if (__syncthreads_or(!landed)) {
            if (tid == 0) {
                const int32_t per_layer = (int32_t)(a.n_tiles * a.n_planes);
                const int32_t l_last = a.layer0 + (int32_t)((blockIdx.x + (n_mine - 1) * gridDim.x) / per_layer);
                for (int32_t l = si.layer; l <= l_last; ++l) atomicOr(&a.err[l], 2);
            }
            timed_out = true;
            break;
        }
        consumed = i + 1;
        if (si.bytes) {
            const uint8_t *stage = ring + (size_t)s * stage_bytes;
            const int32_t rows = si.n * si.heads;
            const uint32_t split = si.order ? (uint32_t)si.heads : (uint32_t)si.n;   // inner extent of a row index
            if (vpr <= kStagedThreads) {
                const int32_t rpp = kStagedThreads / vpr;                  // rows per pass
                const int32_t my = tid / vpr, col = tid - (tid / vpr) * vpr;
                if (my < rpp) {
                    for (int32_t row = my; row < rows; row += rpp * kUnroll) {
                        uint4 v[kUnroll];
                        int64_t off[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const uint32_t r = (uint32_t)(row + u * rpp);
                            if ((int32_t)r < rows) {
                                const uint32_t hi = r / split, lo = r - hi * split;
                                const int64_t h = si.order ? lo : hi, t = si.order ? hi : lo;
                                off[u] = h * a.dst_head_pitch + t * a.dst_pitch + (int64_t)col * 16;
                                v[u] = *reinterpret_cast<const uint4 *>(stage + (size_t)r * a.width + (size_t)col * 16);
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u)
                            if (row + u * rpp < rows) *reinterpret_cast<uint4 *>(si.dst + off[u]) = v[u];
                    }
                }
            } else {
                for (int32_t r = 0; r < rows; ++r) {
                    const uint32_t hi = (uint32_t)r / split, lo = (uint32_t)r - hi * split;
                    const int64_t h = si.order ? lo : hi, t = si.order ? hi : lo;
                    uint8_t *d = si.dst + h * a.dst_head_pitch + t * a.dst_pitch;
                    for (int32_t c = tid; c < vpr; c += kStagedThreads)
                        reinterpret_cast<uint4 *>(d)[c] = reinterpret_cast<const uint4 *>(stage + (size_t)r * a.width)[c];
                }
            }
        }
        __syncthreads();   // every thread has read stage s: it may be refilled
        if (tid == 0 && i + STAGES < n_mine) issue(i + STAGES);
    }
    if (timed_out && tid == 0) {
        // give every load still in flight a bounded chance to land before the ring goes away
        const int64_t issued = n_mine < consumed + STAGES ? n_mine : consumed + STAGES;
        for (int64_t j = consumed; j < issued; ++j) mbar_wait(&bar[j % STAGES], (uint32_t)((j / STAGES) & 1), a.wait_ns);
    }
    stamp_end(a);
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

static cudaError_t resident_grid(const void *fn, int threads, int smem, int per_sm_cap, int *grid, int *sm_count = nullptr) {
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
    if (sm_count) *sm_count = sms;
    return cudaSuccess;
}

template <bool STRIDED, bool TENSOR>
static const void *bulk_fn_of(int stages) {
    switch (stages) {
        case 2: return (const void *)kvx_copy_bulk<2, STRIDED, TENSOR>;
        case 3: return (const void *)kvx_copy_bulk<3, STRIDED, TENSOR>;
        case 6: return (const void *)kvx_copy_bulk<6, STRIDED, TENSOR>;
        case 8: return (const void *)kvx_copy_bulk<8, STRIDED, TENSOR>;
        default: return (const void *)kvx_copy_bulk<4, STRIDED, TENSOR>;
    }
}

static const void *staged_fn(int stages) {
    switch (stages) {
        case 2: return (const void *)kvx_copy_staged<2>;
        case 3: return (const void *)kvx_copy_staged<3>;
        case 6: return (const void *)kvx_copy_staged<6>;
        case 8: return (const void *)kvx_copy_staged<8>;
        default: return (const void *)kvx_copy_staged<4>;
    }
}

static const void *bulk_fn(int stages, bool strided, bool tensor) {
    return tensor ? bulk_fn_of<true, true>(stages) : strided ? bulk_fn_of<true, false>(stages) : bulk_fn_of<false, false>(stages);
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
    if (sh.kernel == KVX_KERNEL_STAGED) {
        const int smem = sh.stages * sh.tile_bytes;
        const bool small = n_work * (int64_t)sh.tile_bytes < ((int64_t)128 << 20);
        const int cap = sh.ctas_per_sm ? sh.ctas_per_sm : (small ? 2 : 64);
        const void *fn = staged_fn(sh.stages);
        e = resident_grid(fn, kStagedThreads, smem, cap, &grid);
        if (e != cudaSuccess) return e;
        if (sh.max_ctas > 0) grid = std::min(grid, sh.max_ctas);
        CopyArgs args_copy = a;
        int64_t work = n_work;
        int32_t stage_bytes = sh.tile_bytes;
        void *args[] = {&args_copy, &work, &stage_bytes};
        return cudaLaunchKernel(fn, dim3((unsigned)std::min<int64_t>(grid, n_work)), dim3(kStagedThreads), args,
                                (size_t)smem, st);
    }
    if (ring_kernel(sh.kernel)) {
        // Launches that read under 128 MiB (a layer push) default to 2 CTAs per SM with a 3-stage
        // ring: measured on GB300, contiguous 64 MiB pushes ran at 0.999 of the copy peak in the
        // per-layer step (consecutive launches overlapping on the lanes) and 0.81 alone, against
        // 0.991 / 0.81 at 1.25 CTAs per SM with 4 stages and 0.94 / 0.85 at 2 per SM with 4 (the
        // deeper ring leaves the next launch no room beside it). TENSOR launches that small take up to
        // 3 CTAs per SM (32 KiB tiles in a 2-stage ring). Larger launches take the occupancy limit.
        // TENSOR stages are 128-byte aligned for the tensor copies.
        const bool tensor = sh.kernel == KVX_KERNEL_TENSOR;
        const int32_t stage_bytes_k = tensor ? (int32_t)align_up((size_t)sh.tile_bytes, 128) : sh.tile_bytes;
        const int smem = sh.stages * stage_bytes_k;
        const bool small = n_work * (int64_t)sh.tile_bytes < ((int64_t)128 << 20);
        const int cap = sh.ctas_per_sm ? sh.ctas_per_sm : (small ? (tensor ? 3 : 2) : 64);
        const void *fn = bulk_fn(sh.stages, sh.strided != 0, tensor);
        int sms = 0;
        e = resident_grid(fn, 32, smem, cap, &grid, &sms);
        if (e != cudaSuccess) return e;
        if (sh.max_ctas > 0) grid = std::min(grid, sh.max_ctas);
        // the fewest CTAs that keep the most items per CTA the same, so every CTA takes as many items
        // (or one fewer) and none starts a round of its own at the end. Measured on GB300, 32 MiB
        // head-layout pushes (1024 tiles of 32 KiB): 342 CTAs of 3 tiles 0.954-0.955 of the copy peak
        // in the per-layer step and 0.714 alone, against 456 CTAs (3 per SM, 2.25 tiles each) 0.90 /
        // 0.69 and 304 (2 per SM) 0.928 / 0.665; contiguous 64 MiB pushes (2048 tiles): 293 CTAs 0.987
        // / 0.805 against 304 CTAs 0.987 / 0.803.
        if (grid > 0 && n_work > 0) {
            const int64_t per = (n_work + grid - 1) / grid;
            grid = (int)((n_work + per - 1) / per);
        }
        CopyArgs args_copy = a;
        int64_t work = n_work;
        int32_t stage_bytes = stage_bytes_k;
        // evict-first L2 hints for contiguous and tensor-map launches that stream at least
        // kStreamL2Bytes. Smaller ones keep the default policy (a 1 MB push whose blocks stay in L2
        // between steps ran 7 % slower with it), and so do strided row-by-row ones: rows written
        // one by one into lines that other items complete later ran 6-7 % slower with it
        // (fragmented head-group pushes, 32 MiB per layer), 512-byte remap rows gained under 1 %.
        int32_t stream_l2 = (!sh.strided || tensor) && n_work * (int64_t)sh.tile_bytes >= kStreamL2Bytes;
        void *args[] = {&args_copy, &work, &stage_bytes, &stream_l2};
        return cudaLaunchKernel(fn, dim3((unsigned)std::min<int64_t>(grid, n_work)), dim3(32), args, (size_t)smem, st);
    }
    // default resident CTAs: small launches stay small so that they overlap the caller's compute and
    // the next push (head-group tiles, many short rows each, at 4 per SM: 0.81 of the copy peak at
    // 128 threads against 0.75 at 8 and 12 on 32 MiB-per-layer pushes); large ones take the whole GPU
    LaunchShape shape = sh;
    if (shape.ctas_per_sm == 0)
        shape.ctas_per_sm = n_work * (int64_t)sh.tile_bytes < ((int64_t)128 << 20) ? (sh.head_groups ? 4 : 2) : 64;
    if (sh.kernel == KVX_KERNEL_PERSIST) {
        const void *fn = sh.vec == 16 ? persist_fn<16>(sh.strided) : sh.vec == 8 ? persist_fn<8>(sh.strided)
                       : sh.vec == 4 ? persist_fn<4>(sh.strided) : sh.vec == 2 ? persist_fn<2>(sh.strided)
                       : persist_fn<1>(sh.strided);
        e = resident_grid(fn, sh.threads, 0, shape.ctas_per_sm, &grid);
        if (e != cudaSuccess) return e;
        if (sh.max_ctas > 0) grid = std::min(grid, sh.max_ctas);
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

}  // namespace kvx
