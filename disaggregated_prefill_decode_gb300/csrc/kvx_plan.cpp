// Host side of kvx: error reporting, plan validation and the plan API. The runs, tiles and launch
// shape a plan gets are built in kvx_tiles.cpp. No device work.
//
// Follows the push-mode NIXL connector article (spke.com 3844), section "Threading-Modell" (block ids
// are mapped to memory descriptors and contiguous blocks merged into larger regions) and
// "Implementierungsdetails" step 3 (each side maps block positions to its own layout), and the
// "vLLM MoRIIO KV Connector" notes, section 6 (transfer triples with adjacent blocks merged; rank
// mapping when one TP size is a multiple of the other).
#include "kvx_internal.h"

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <new>
#include <numeric>

namespace kvx {

static thread_local char g_err[512] = "";
static std::atomic<int64_t> g_launches{0};

kvx_status fail(kvx_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

kvx_status cuda_fail(cudaError_t e, const char *what) {
    return fail(KVX_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void count_launch(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static kvx_status read_geom(const kvx_pool *p, const char *side, Geom *g, std::vector<void *> *bases) {
    if (!p) return fail(KVX_EINVAL, "%s pool is NULL", side);
    if (p->n_layers < 1 || p->n_planes < 1 || p->n_shards < 1 || p->heads_per_shard < 1 || p->head_dim < 1 ||
        p->elem_bytes < 1 || p->block_size < 1 || p->n_blocks < 0)
        return fail(KVX_EINVAL, "%s pool: counts must be >= 1 (n_blocks >= 0)", side);
    if (p->layout != KVX_LAYOUT_NHD && p->layout != KVX_LAYOUT_HND)
        return fail(KVX_EUNSUPPORTED, "%s pool: unknown layout %d", side, p->layout);
    *g = Geom{p->n_layers, p->n_planes, p->n_shards, p->heads_per_shard, p->head_dim, p->elem_bytes,
              p->block_size, p->layout, p->n_blocks};
    // extents stay well inside int64, rows inside int32, buffers inside the int32 launch grid
    const double bytes = (double)p->n_blocks * p->block_size * p->heads_per_shard * (double)p->head_dim * p->elem_bytes;
    if (bytes > 9.0e18) return fail(KVX_EUNSUPPORTED, "%s pool buffer size overflows", side);
    if ((double)p->n_blocks * p->block_size > (double)std::numeric_limits<int32_t>::max())
        return fail(KVX_EUNSUPPORTED, "%s pool has more than 2^31-1 rows per buffer", side);
    if ((double)p->n_layers * p->n_planes * p->n_shards > 1.0e7)
        return fail(KVX_EUNSUPPORTED, "%s pool has too many buffers", side);
    if (p->n_layers > 65535 || p->n_planes > 65535)
        return fail(KVX_EUNSUPPORTED, "%s pool: at most 65535 layers and planes", side);
    if (!p->base) return fail(KVX_EINVAL, "%s pool base table is NULL", side);
    const int32_t n = g->n_buffers();
    bases->assign(p->base, p->base + n);
    for (int32_t i = 0; i < n; ++i)
        if (!(*bases)[i] && g->buf_bytes() > 0) return fail(KVX_EINVAL, "%s pool buffer %d is NULL", side, i);
    return KVX_OK;
}

// A consumer buffer that overlaps a producer buffer or another consumer buffer makes the copy a race.
static kvx_status check_overlap(const std::vector<void *> &src, int64_t src_bytes, const std::vector<void *> &dst,
                                int64_t dst_bytes) {
    struct Iv { uintptr_t lo, hi; int dst; };
    std::vector<Iv> iv;
    iv.reserve(src.size() + dst.size());
    if (src_bytes > 0)
        for (void *p : src) iv.push_back({(uintptr_t)p, (uintptr_t)p + (uintptr_t)src_bytes, 0});
    if (dst_bytes > 0)
        for (void *p : dst) iv.push_back({(uintptr_t)p, (uintptr_t)p + (uintptr_t)dst_bytes, 1});
    std::sort(iv.begin(), iv.end(), [](const Iv &a, const Iv &b) { return a.lo < b.lo; });
    // sweep in address order, remembering the furthest end of consumer and producer intervals seen
    uintptr_t max_dst_hi = 0, max_src_hi = 0;
    bool any_dst = false, any_src = false;
    for (const Iv &v : iv) {
        if (any_dst && v.lo < max_dst_hi) return fail(KVX_EINVAL, "a consumer buffer overlaps another pool buffer");
        if (v.dst && any_src && v.lo < max_src_hi) return fail(KVX_EINVAL, "a consumer buffer overlaps a producer buffer");
        if (v.dst) { max_dst_hi = std::max(max_dst_hi, v.hi); any_dst = true; }
        else { max_src_hi = std::max(max_src_hi, v.hi); any_src = true; }
    }
    return KVX_OK;
}


// Default lane count: 4, or half the hardware work queues the CUDA runtime gave this process when
// that is fewer (CUDA_DEVICE_MAX_CONNECTIONS as the process started, 8 when unset; at least 1).
// Streams beyond the queues share them, and a lane that shares one with the caller's compute stream
// or another lane waits behind its work (a false dependency). Measured on GB300, per-layer pushes of
// 64 MiB overlapping on the lanes, fraction of the copy peak contiguous / head-layout change: with
// 8 queues 4 lanes 0.984 / 0.92-0.93, 8 lanes 0.965 / 0.88; with 32 queues 4 lanes 0.985 / 0.92-0.93,
// 8 lanes 0.993 / 0.955, but the per-layer step (pushes beside a short prefill) then took 0.67-0.69 ms
// against 0.64-0.65 (the extra concurrent copies stretch the prefill chain) and the end-to-end path
// from host memory fell from 303 to 272 GB/s; 6 lanes ran 497 MB layers at 0.86-0.87 against 1.01.
int32_t default_lanes() {
    static const int32_t lanes = [] {
        const char *e = std::getenv("CUDA_DEVICE_MAX_CONNECTIONS");
        char *end = nullptr;
        long queues = e ? std::strtol(e, &end, 10) : 8;
        if (!e || end == e || queues < 1) queues = 8;       // unset or not a count: the runtime's default
        return (int32_t)std::max<long>(1, std::min<long>(4, queues / 2));
    }();
    return lanes;
}

kvx_status init_plan_geometry(const kvx_pool *src, const kvx_pool *dst, const kvx_plan_opts *opts, kvx_plan_s *pl) {
    pl->lanes = default_lanes();
    kvx_status st = read_geom(src, "producer", &pl->src, &pl->src_base);
    if (st) return st;
    st = read_geom(dst, "consumer", &pl->dst, &pl->dst_base);
    if (st) return st;
    const Geom &s = pl->src, &d = pl->dst;
    if (s.n_layers != d.n_layers || s.n_planes != d.n_planes)
        return fail(KVX_EINVAL, "layer/plane counts differ (%d x %d vs %d x %d)", s.n_layers, s.n_planes,
                    d.n_layers, d.n_planes);
    if (s.head_dim != d.head_dim || s.elem_bytes != d.elem_bytes) return fail(KVX_EINVAL, "head_dim / elem_bytes differ");
    if ((int64_t)s.n_shards * s.heads_per_shard != (int64_t)d.n_shards * d.heads_per_shard)
        return fail(KVX_EINVAL, "total KV heads differ (%d vs %d)", s.n_shards * s.heads_per_shard,
                    d.n_shards * d.heads_per_shard);
    if (std::max(s.n_shards, d.n_shards) % std::min(s.n_shards, d.n_shards) != 0)
        return fail(KVX_EUNSUPPORTED, "shard counts %d and %d do not divide one another", s.n_shards, d.n_shards);
    st = check_overlap(pl->src_base, s.buf_bytes(), pl->dst_base, d.buf_bytes());
    if (st) return st;
    if (opts) {
        if (opts->layers_per_launch < 0) return fail(KVX_EINVAL, "layers_per_launch must be >= 0");
        if (!valid_stages(opts->bulk_stages)) return fail(KVX_EINVAL, "bulk_stages must be 0, 2, 3, 4, 6 or 8");
        if (opts->flags & ~KVX_PLAN_TIMING) return fail(KVX_EINVAL, "unknown kvx_plan_opts.flags bits");
        if (opts->tile_bytes) pl->tile_bytes = opts->tile_bytes;
        if (opts->threads) pl->threads = opts->threads;
        pl->threads_req = opts->threads;
        pl->flags = opts->flags;
        if (opts->kernel < 0 || opts->kernel > KVX_KERNEL_STAGED) return fail(KVX_EINVAL, "unknown kernel %d", opts->kernel);
        if (opts->max_ctas < 0) return fail(KVX_EINVAL, "max_ctas must be >= 0");
        pl->max_ctas = opts->max_ctas;
        if (opts->ctas_per_sm < 0 || opts->ctas_per_sm > 64) return fail(KVX_EINVAL, "ctas_per_sm in [0, 64]");
        if (opts->lanes < 0 || opts->lanes > 8) return fail(KVX_EINVAL, "lanes in [0, 8]");
        pl->kernel = opts->kernel;
        if (opts->ctas_per_sm) pl->ctas_per_sm = opts->ctas_per_sm;
        if (opts->lanes) pl->lanes = opts->lanes;
        pl->bulk_stages_req = opts->bulk_stages;
        pl->layers_per_launch_req = opts->layers_per_launch;
    }
    if (pl->tile_bytes < 16 || pl->tile_bytes % 16 || pl->tile_bytes > (1 << 26))
        return fail(KVX_EINVAL, "tile_bytes must be a multiple of 16 in [16, 2^26]");
    if (pl->threads < 32 || pl->threads > 1024 || pl->threads % 32)
        return fail(KVX_EINVAL, "threads must be a multiple of 32 in [32, 1024]");
    init_copy_shape(pl, opts && opts->tile_bytes);
    pl->layer_state.assign(s.n_layers, KVX_LAYER_IDLE);
    pl->inject.assign(s.n_layers, 0);
    pl->injected_pending.assign(s.n_layers, 0);
    pl->stall.assign(s.n_layers, 0);
    return KVX_OK;
}

}  // namespace kvx

using namespace kvx;

extern "C" {

const char *kvx_status_str(kvx_status s) {
    switch (s) {
        case KVX_OK: return "KVX_OK";
        case KVX_EINVAL: return "KVX_EINVAL";
        case KVX_ERANGE: return "KVX_ERANGE";
        case KVX_EOVERLAP: return "KVX_EOVERLAP";
        case KVX_EUNSUPPORTED: return "KVX_EUNSUPPORTED";
        case KVX_ENOMEM: return "KVX_ENOMEM";
        case KVX_ECUDA: return "KVX_ECUDA";
        case KVX_ETIMEDOUT: return "KVX_ETIMEDOUT";
        case KVX_EFAILED: return "KVX_EFAILED";
    }
    return "KVX_UNKNOWN";
}

const char *kvx_last_error(void) { return g_err; }

const char *kvx_version(void) { return "kvx 0.1 (sm_103a)"; }

int64_t kvx_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

kvx_status kvx_plan_ex(const kvx_pool *src, const kvx_pool *dst, const kvx_request *reqs, int32_t n_reqs,
                       const kvx_plan_opts *opts, kvx_plan_t *out) {
    if (!out) return fail(KVX_EINVAL, "out is NULL");
    *out = nullptr;
    if (n_reqs < 0 || (n_reqs > 0 && !reqs)) return fail(KVX_EINVAL, "bad request array");
    kvx_plan_s *pl = new (std::nothrow) kvx_plan_s();
    if (!pl) return fail(KVX_ENOMEM, "host allocation failed");
    kvx_status st = init_plan_geometry(src, dst, opts, pl);
    if (st) { delete pl; return st; }
    const Geom &s = pl->src, &d = pl->dst;

    // requests: counts, id ranges, consumer blocks used once
    std::vector<uint8_t> used((size_t)d.n_blocks, 0);
    for (int32_t r = 0; r < n_reqs; ++r) {
        const kvx_request &q = reqs[r];
        if (q.n_tokens < 0) { delete pl; return fail(KVX_EINVAL, "request %d: n_tokens < 0", r); }
        const int64_t ns = ceil_div(q.n_tokens, s.block_size), nd = ceil_div(q.n_tokens, d.block_size);
        if (q.n_src < ns || q.n_dst < nd) {
            delete pl;
            return fail(KVX_ERANGE, "request %d: %lld tokens need %lld producer and %lld consumer ids (got %d, %d)", r,
                        (long long)q.n_tokens, (long long)ns, (long long)nd, q.n_src, q.n_dst);
        }
        if ((ns > 0 && !q.src_block_ids) || (nd > 0 && !q.dst_block_ids)) {
            delete pl;
            return fail(KVX_EINVAL, "request %d: id array is NULL", r);
        }
        for (int64_t i = 0; i < ns; ++i)
            if (q.src_block_ids[i] < 0 || q.src_block_ids[i] >= s.n_blocks) {
                delete pl;
                return fail(KVX_ERANGE, "request %d: producer block id %d outside [0, %lld)", r, q.src_block_ids[i],
                            (long long)s.n_blocks);
            }
        for (int64_t i = 0; i < nd; ++i) {
            const int32_t b = q.dst_block_ids[i];
            if (b < 0 || b >= d.n_blocks) {
                delete pl;
                return fail(KVX_ERANGE, "request %d: consumer block id %d outside [0, %lld)", r, b, (long long)d.n_blocks);
            }
            if (used[(size_t)b]) {
                delete pl;
                return fail(KVX_EOVERLAP, "request %d: consumer block %d is written twice", r, b);
            }
            used[(size_t)b] = 1;
        }
    }
    for (int32_t r = 0; r < n_reqs; ++r)
        request_runs(reqs[r].n_tokens, s.block_size, reqs[r].src_block_ids, d.block_size, reqs[r].dst_block_ids, pl);
    finish_plan_shape(pl);
    build_tiles(pl);
    if (pl->n_tiles > std::numeric_limits<int32_t>::max()) {
        delete pl;
        return fail(KVX_EUNSUPPORTED, "plan needs more than 2^31-1 tiles per layer; raise tile_bytes");
    }
    *out = pl;
    return KVX_OK;
}

kvx_status kvx_plan(const kvx_pool *src, const kvx_pool *dst, const kvx_request *reqs, int32_t n_reqs,
                    kvx_plan_t *out) {
    return kvx_plan_ex(src, dst, reqs, n_reqs, nullptr, out);
}

kvx_status kvx_plan_set_opts(kvx_plan_t pl, const kvx_plan_opts *o) {
    if (!pl || !o) return fail(KVX_EINVAL, "NULL argument");
    if (!pl->pending.empty()) return fail(KVX_EINVAL, "pushes are pending; kvx_sync first");
    if (o->tile_bytes && o->tile_bytes != pl->tile_bytes) return fail(KVX_EINVAL, "tile_bytes is fixed once tiles exist");
    if (o->layers_per_launch < 0) return fail(KVX_EINVAL, "layers_per_launch must be >= 0");
    if (!valid_stages(o->bulk_stages)) return fail(KVX_EINVAL, "bulk_stages must be 0, 2, 3, 4, 6 or 8");
    if (o->flags & ~KVX_PLAN_TIMING) return fail(KVX_EINVAL, "unknown kvx_plan_opts.flags bits");
    if (o->kernel < 0 || o->kernel > KVX_KERNEL_STAGED) return fail(KVX_EINVAL, "unknown kernel %d", o->kernel);
    if (o->max_ctas < 0) return fail(KVX_EINVAL, "max_ctas must be >= 0");
    if (o->ctas_per_sm < 0 || o->ctas_per_sm > 64) return fail(KVX_EINVAL, "ctas_per_sm in [0, 64]");
    if (o->lanes < 0 || o->lanes > 8) return fail(KVX_EINVAL, "lanes in [0, 8]");
    if (o->threads && (o->threads < 32 || o->threads > 1024 || o->threads % 32))
        return fail(KVX_EINVAL, "threads must be a multiple of 32 in [32, 1024]");
    pl->flags = o->flags;
    if (o->threads) pl->threads = o->threads;
    pl->threads_req = o->threads;
    pl->ctas_per_sm = o->ctas_per_sm;
    pl->lanes = o->lanes ? o->lanes : default_lanes();
    pl->bulk_stages_req = o->bulk_stages;
    pl->layers_per_launch_req = o->layers_per_launch;
    pl->max_ctas = o->max_ctas;
    pl->next_lane = 0;
    pl->lane_cache.clear();
    pl->lane_src = nullptr;
    pl->kernel = o->kernel;
    resolve_launch(pl);
    return KVX_OK;
}

kvx_status kvx_plan_runs(kvx_plan_t pl, int64_t *n_runs, const int32_t **src_row, const int32_t **dst_row,
                         const int32_t **n_tokens) {
    if (!pl || !n_runs) return fail(KVX_EINVAL, "NULL argument");
    if (pl->n_runs_dev > 0 && pl->run_ntok.empty()) {
        // a device-built plan's runs stay on the device until asked for (the kernels that wrote
        // them finished before kvx_match_prefix returned)
        const size_t n = (size_t)pl->n_runs_dev;
        std::vector<int32_t> s(n), d(n), t(n);
        const int32_t *rows = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(pl->dev) + pl->off_runs);
        cudaError_t e = cudaMemcpy(s.data(), rows, sizeof(int32_t) * n, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(d.data(), rows + pl->run_cap, sizeof(int32_t) * n, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(t.data(), rows + 2 * pl->run_cap, sizeof(int32_t) * n, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "reading plan runs");
        pl->run_src_row.swap(s);
        pl->run_dst_row.swap(d);
        pl->run_ntok.swap(t);
    }
    *n_runs = (int64_t)pl->run_ntok.size();
    if (src_row) *src_row = pl->run_src_row.data();
    if (dst_row) *dst_row = pl->run_dst_row.data();
    if (n_tokens) *n_tokens = pl->run_ntok.data();
    return KVX_OK;
}

kvx_status kvx_plan_get_info(kvx_plan_t pl, kvx_plan_info *out) {
    if (!pl || !out) return fail(KVX_EINVAL, "NULL argument");
    out->n_runs = pl->n_runs_dev >= 0 ? pl->n_runs_dev : (int64_t)pl->run_ntok.size();
    out->n_tiles = pl->n_tiles;
    out->bytes_per_layer = pl->bytes_per_layer;
    out->vec_bytes = pl->vec;
    out->strided = pl->strided;
    out->n_layers = pl->src.n_layers;
    out->n_planes = pl->src.n_planes;
    out->width = pl->width;
    out->tile_bytes = pl->tile_bytes;
    const int32_t k = effective_kernel(pl);
    out->kernel = k;
    out->threads = ring_kernel(k) ? 32 : staged_kernel(k) ? 128 : pl->threads;
    out->lanes = pl->lanes;
    out->bulk_stages = ring_kernel(k) || staged_kernel(k) ? pl->bulk_stages : 0;
    out->src_pitch = pl->src_pitch;
    out->dst_pitch = pl->dst_pitch;
    out->src_head_pitch = pl->src_head_pitch;
    out->dst_head_pitch = pl->dst_head_pitch;
    return KVX_OK;
}

kvx_status kvx_plan_tiles(kvx_plan_t pl, int64_t *n_tiles, const void **tiles) {
    if (!pl || !n_tiles || !tiles) return fail(KVX_EINVAL, "NULL argument");
    *n_tiles = (int64_t)pl->tiles.size();
    *tiles = pl->tiles.data();
    return KVX_OK;
}

kvx_status kvx_plan_push_times(kvx_plan_t pl, float *start_us, float *end_us, int32_t cap, int32_t *n) {
    if (!pl || !n || (cap > 0 && (!start_us || !end_us))) return fail(KVX_EINVAL, "NULL argument");
    if (!(pl->flags & KVX_PLAN_TIMING)) return fail(KVX_EINVAL, "plan was built without KVX_PLAN_TIMING");
    *n = (int32_t)pl->push_start_us.size();
    for (int32_t i = 0; i < *n && i < cap; ++i) {
        start_us[i] = pl->push_start_us[i];
        end_us[i] = pl->push_end_us[i];
    }
    return KVX_OK;
}

kvx_status kvx_plan_push_times_ns(kvx_plan_t pl, int64_t *start_ns, int64_t *end_ns, int32_t cap, int32_t *n) {
    if (!pl || !n || (cap > 0 && (!start_ns || !end_ns))) return fail(KVX_EINVAL, "NULL argument");
    if (!(pl->flags & KVX_PLAN_TIMING)) return fail(KVX_EINVAL, "plan was built without KVX_PLAN_TIMING");
    *n = (int32_t)pl->push_start_ns.size();
    for (int32_t i = 0; i < *n && i < cap; ++i) {
        start_ns[i] = pl->push_start_ns[i];
        end_ns[i] = pl->push_end_ns[i];
    }
    return KVX_OK;
}

kvx_status kvx_plan_layer_states(kvx_plan_t pl, int32_t *out, int32_t n_layers) {
    if (!pl || !out) return fail(KVX_EINVAL, "NULL argument");
    if (n_layers != pl->src.n_layers) return fail(KVX_EINVAL, "plan has %d layers", pl->src.n_layers);
    for (int32_t l = 0; l < n_layers; ++l) out[l] = pl->layer_state[l];
    return KVX_OK;
}

kvx_status kvx_plan_inject_failure(kvx_plan_t pl, int32_t layer) {
    if (!pl) return fail(KVX_EINVAL, "NULL plan");
    if (layer < 0 || layer >= pl->src.n_layers) return fail(KVX_EINVAL, "layer %d out of range", layer);
    pl->inject[layer] = 1;
    return KVX_OK;
}

kvx_status kvx_plan_inject_stall(kvx_plan_t pl, int32_t layer) {
    if (!pl) return fail(KVX_EINVAL, "NULL plan");
    if (layer < 0 || layer >= pl->src.n_layers) return fail(KVX_EINVAL, "layer %d out of range", layer);
    const int32_t k = effective_kernel(pl);
    if (!ring_kernel(k) && !staged_kernel(k))
        return fail(KVX_EUNSUPPORTED, "the stall hook needs a plan whose pushes run a shared-memory ring kernel");
    pl->stall[layer] = 1;
    return KVX_OK;
}

}  // extern "C"
