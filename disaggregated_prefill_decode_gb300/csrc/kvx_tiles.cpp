// The copy shape of a plan, on the host: merged token runs, head-shard pairs, the vector width, the
// tile tables (contiguous, strided, per head), the default tile size and the kernel / ring choice.
// No device work. Everything here decides what the copy kernels are given.
//
// Follows the push-mode NIXL connector article (spke.com 3844), section "Threading-Modell" (block ids
// are mapped to memory descriptors and contiguous blocks merged into larger regions) and
// "Implementierungsdetails" step 3 (each side maps block positions to its own layout), and the
// "vLLM MoRIIO KV Connector" notes, section 6 (transfer triples with adjacent blocks merged; rank
// mapping when one TP size is a multiple of the other).
#include "kvx_internal.h"

#include <algorithm>
#include <numeric>

namespace kvx {

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Appends the maximal token runs of one request. Walks the segments between consecutive block
// boundaries of either side (rows inside a segment advance together), and extends the previous run
// when both sides continue it.
void request_runs(int64_t n_tok, int32_t bs_s, const int32_t *sids, int32_t bs_d, const int32_t *dids,
                  kvx_plan_s *pl) {
    const size_t first = pl->run_ntok.size();
    int64_t t = 0;
    while (t < n_tok) {
        const int64_t is = t / bs_s, id = t / bs_d;
        const int64_t end = std::min({(is + 1) * bs_s, (id + 1) * bs_d, n_tok});
        const int64_t srow = (int64_t)sids[is] * bs_s + (t - is * bs_s);
        const int64_t drow = (int64_t)dids[id] * bs_d + (t - id * bs_d);
        const int32_t len = (int32_t)(end - t);
        const size_t k = pl->run_ntok.size();
        if (k > first && (int64_t)pl->run_src_row[k - 1] + pl->run_ntok[k - 1] == srow &&
            (int64_t)pl->run_dst_row[k - 1] + pl->run_ntok[k - 1] == drow) {
            pl->run_ntok[k - 1] += len;
        } else {
            pl->run_src_row.push_back((int32_t)srow);
            pl->run_dst_row.push_back((int32_t)drow);
            pl->run_ntok.push_back(len);
        }
        t = end;
    }
}

// Head-shard pairs: the contiguous head ranges that one producer shard and one consumer shard share.
std::vector<Pair> shard_pairs(const Geom &s, const Geom &d) {
    std::vector<Pair> out;
    const int64_t hb = s.head_bytes();
    if (s.heads_per_shard == d.heads_per_shard) {
        for (int32_t i = 0; i < s.n_shards; ++i) out.push_back({i, i, 0, 0});
    } else if (s.heads_per_shard < d.heads_per_shard) {   // merge: several producer shards per consumer shard
        for (int32_t i = 0; i < s.n_shards; ++i) {
            const int32_t g0 = i * s.heads_per_shard;
            const int32_t ds = g0 / d.heads_per_shard;
            out.push_back({i, ds, 0, (int64_t)(g0 - ds * d.heads_per_shard) * hb});
        }
    } else {                                              // split: several consumer shards per producer shard
        for (int32_t j = 0; j < d.n_shards; ++j) {
            const int32_t g0 = j * d.heads_per_shard;
            const int32_t ss = g0 / s.heads_per_shard;
            out.push_back({ss, j, (int64_t)(g0 - ss * s.heads_per_shard) * hb, 0});
        }
    }
    return out;
}

static int64_t gcd64(int64_t a, int64_t b) { return std::gcd(a < 0 ? -a : a, b < 0 ? -b : b); }

// The widest vector (<= 16 bytes) dividing every address, offset and length the copy uses.
static int32_t vector_bytes(const kvx_plan_s *pl, const std::vector<Pair> &pairs) {
    int64_t g = 16;
    for (void *p : pl->src_base) g = gcd64(g, (int64_t)((uintptr_t)p & 15));
    for (void *p : pl->dst_base) g = gcd64(g, (int64_t)((uintptr_t)p & 15));
    g = gcd64(g, pl->src.row_bytes());
    g = gcd64(g, pl->dst.row_bytes());
    if (pl->per_head) {
        g = gcd64(g, pl->src.head_bytes());   // offsets, pitches and widths are multiples of it
    } else if (pl->strided) {
        g = gcd64(g, pl->width);
        for (const Pair &q : pairs) g = gcd64(gcd64(g, q.src_seg_off), q.dst_seg_off);
    } else {
        g = gcd64(g, pl->tile_bytes);
    }
    return (int32_t)g;   // gcd with 16: one of 16, 8, 4, 2, 1
}

// Tiles of plans with an HND side: each run is cut at every block boundary of either side, and each
// such segment is copied by groups of heads (a head's tokens are rows at each side's token pitch, and
// the heads of a group, consecutive heads that one producer shard and one consumer shard share, are
// a head pitch apart on each side): as many heads per tile as fit tile_bytes. When both sides are
// HND with the same block size and heads per shard, a stretch of whole blocks is one contiguous span
// per shard on both sides and is copied as such.
static bool same_head_major(const Geom &s, const Geom &d) {
    return s.layout == KVX_LAYOUT_HND && d.layout == KVX_LAYOUT_HND && s.block_size == d.block_size &&
           s.heads_per_shard == d.heads_per_shard;
}

static void build_head_tiles(kvx_plan_s *pl) {
    const Geom &s = pl->src, &d = pl->dst;
    const int64_t hb = s.head_bytes();
    const int64_t rows_per_tile = std::max<int64_t>(1, pl->tile_bytes / hb);
    const int32_t heads = s.n_shards * s.heads_per_shard;
    const bool same_hnd = same_head_major(s, d);
    auto emit = [&](int64_t soff, int64_t doff, int64_t rows, int32_t ss, int32_t ds) {
        for (int64_t r0 = 0; r0 < rows; r0 += rows_per_tile)
            pl->tiles.push_back({soff + r0 * pl->src_pitch, doff + r0 * pl->dst_pitch,
                                 (int32_t)std::min(rows_per_tile, rows - r0), ss, ds, 0});
    };
    for (size_t r = 0; r < pl->run_ntok.size(); ++r) {
        int64_t t = 0;
        const int64_t n = pl->run_ntok[r];
        while (t < n) {
            const int64_t srow = (int64_t)pl->run_src_row[r] + t, drow = (int64_t)pl->run_dst_row[r] + t;
            const int64_t sblk = srow / s.block_size, sslot = srow % s.block_size;
            const int64_t dblk = drow / d.block_size, dslot = drow % d.block_size;
            if (same_hnd && sslot == 0 && dslot == 0 && n - t >= s.block_size) {
                const int64_t nblk = (n - t) / s.block_size;        // whole blocks, contiguous on both sides
                for (int32_t sh = 0; sh < s.n_shards; ++sh)
                    emit(s.head_index(sblk, 0, 0) * hb, d.head_index(dblk, 0, 0) * hb,
                         nblk * s.block_size * s.heads_per_shard, sh, sh);
                t += nblk * s.block_size;
                continue;
            }
            const int64_t len = std::min({s.block_size - sslot, d.block_size - dslot, n - t});
            const int64_t per_tile = std::max<int64_t>(1, rows_per_tile / len);      // heads per tile
            for (int32_t g = 0; g < heads;) {
                const int32_t ss = g / s.heads_per_shard, hs = g % s.heads_per_shard;
                const int32_t ds = g / d.heads_per_shard, hd = g % d.heads_per_shard;
                const int32_t k = (int32_t)std::min<int64_t>({per_tile, s.heads_per_shard - hs, d.heads_per_shard - hd});
                const int64_t so = s.head_index(sblk, sslot, hs) * hb, dof = d.head_index(dblk, dslot, hd) * hb;
                if (k == 1)
                    emit(so, dof, len, ss, ds);
                else
                    pl->tiles.push_back({so, dof, (int32_t)len, ss, ds, k});
                g += k;
            }
            t += len;
        }
    }
    pl->n_tiles = (int64_t)pl->tiles.size();
}

void build_tiles(kvx_plan_s *pl) {
    const std::vector<Pair> pairs = shard_pairs(pl->src, pl->dst);
    pl->tiles.clear();
    if (pl->per_head) {
        build_head_tiles(pl);
        return;
    }
    const int64_t rb_s = pl->src.row_bytes(), rb_d = pl->dst.row_bytes();
    const size_t nr = pl->run_ntok.size();
    if (!pl->strided) {
        for (size_t r = 0; r < nr; ++r) {
            const int64_t bytes = (int64_t)pl->run_ntok[r] * rb_s;
            const int64_t s0 = (int64_t)pl->run_src_row[r] * rb_s, d0 = (int64_t)pl->run_dst_row[r] * rb_d;
            for (int64_t o = 0; o < bytes; o += pl->tile_bytes)
                for (const Pair &q : pairs)
                    pl->tiles.push_back({s0 + o, d0 + o, (int32_t)std::min<int64_t>(pl->tile_bytes, bytes - o),
                                         q.s, q.d, 0});
        }
    } else {
        const int64_t rpt = std::max<int64_t>(1, pl->tile_bytes / pl->width);
        for (size_t r = 0; r < nr; ++r)
            for (int64_t r0 = 0; r0 < pl->run_ntok[r]; r0 += rpt) {
                const int32_t rows = (int32_t)std::min<int64_t>(rpt, pl->run_ntok[r] - r0);
                for (const Pair &q : pairs)
                    pl->tiles.push_back({((int64_t)pl->run_src_row[r] + r0) * rb_s + q.src_seg_off,
                                         ((int64_t)pl->run_dst_row[r] + r0) * rb_d + q.dst_seg_off, rows, q.s, q.d, 0});
            }
    }
    pl->n_tiles = (int64_t)pl->tiles.size();
}

// Default tile of a contiguous plan. Runs are cut at the block boundaries of both sides, so the usual
// run is a whole number of "units" of min(block sizes) token rows. A unit above 16 KiB is split into
// the fewest equal tiles of at most 16 KiB (a 36,864-byte MLA block: 3 x 12 KiB rather than
// 16 + 16 + 4 KiB, whose short tail wastes a bulk-ring stage); smaller units are packed whole.
static int32_t default_tile_bytes(const Geom &s, const Geom &d) {
    constexpr int64_t kTarget = 16384;
    const int64_t unit = (int64_t)std::min(s.block_size, d.block_size) * s.row_bytes();
    int64_t t;
    if (unit >= kTarget) {
        const int64_t k = ceil_div(unit, kTarget);
        t = ceil_div(unit, k);
        t = ceil_div(t, 16) * 16;
        if (t > kTarget) t = kTarget;
    } else {
        t = unit * std::max<int64_t>(1, kTarget / unit);
    }
    return (int32_t)std::max<int64_t>(16, t - t % 16);
}

// Default tile of a plan that maps one head layout onto another: a segment of min(block sizes)
// tokens for the most heads a producer shard and a consumer shard share that fit `target` bytes, the
// head count a divisor of the shared group so that every group splits into equal tiles (each then
// one tensor-map box; see tensor_box). The target is kHeadTileTarget, or kTensorTileTarget for plans
// that resolve to TENSOR (measured on GB300, 32 MiB per layer in the per-layer step, a consumer or
// producer side moved by plain bulk copies, 2 CTAs per SM: 16 KiB tiles in a 4-stage ring 0.886-0.888
// of the copy peak, 32 KiB tiles -- a whole block of 8 heads -- in a 2-stage ring 0.922-0.931, in a
// 3-stage ring 0.85; alone 0.65-0.68 against 0.665 and 0.72; the 2-stage ring of 32 KiB tiles at up to
// 3 CTAs per SM with every CTA taking 3 tiles: 0.954-0.958, alone 0.712).
constexpr int64_t kHeadTileTarget = 16384;
constexpr int64_t kTensorTileTarget = 32768;

static int32_t default_head_tile_bytes(const Geom &s, const Geom &d, int64_t target) {
    const int64_t hb = s.head_bytes();
    const int64_t n = std::min(s.block_size, d.block_size);
    const int32_t group = std::min(s.heads_per_shard, d.heads_per_shard);
    int32_t k = 1;
    for (int32_t c = group; c >= 1; --c)
        if (group % c == 0 && c * n * hb <= target) { k = c; break; }
    const int64_t t = std::max<int64_t>(16, std::min<int64_t>((int64_t)k * n * hb, target));
    return (int32_t)(t - t % 16);
}

// Copy shape from the two geometries: head-major sides copy per (block segment, head), unequal head
// partitions copy strided rows of the shared head range, and the rest copies contiguous bytes.
void init_copy_shape(kvx_plan_s *pl, bool tile_bytes_given) {
    const Geom &s = pl->src, &d = pl->dst;
    pl->per_head = (s.layout == KVX_LAYOUT_HND || d.layout == KVX_LAYOUT_HND) ? 1 : 0;
    pl->strided = (pl->per_head || s.heads_per_shard != d.heads_per_shard) ? 1 : 0;
    pl->width = (int32_t)(pl->per_head ? s.head_bytes() : std::min(s.heads_per_shard, d.heads_per_shard) * s.head_bytes());
    pl->src_pitch = pl->per_head ? s.token_pitch() : s.row_bytes();
    pl->dst_pitch = pl->per_head ? d.token_pitch() : d.row_bytes();
    // per-head plans: from a head to the next inside one shard, at the same token
    pl->src_head_pitch = pl->per_head ? (s.layout == KVX_LAYOUT_HND ? s.block_size : 1) * s.head_bytes() : 0;
    pl->dst_head_pitch = pl->per_head ? (d.layout == KVX_LAYOUT_HND ? d.block_size : 1) * d.head_bytes() : 0;
    if (!tile_bytes_given && !pl->strided) pl->tile_bytes = default_tile_bytes(s, d);
    pl->head_tile_auto = !tile_bytes_given && pl->per_head && !same_head_major(s, d);
    if (pl->head_tile_auto) pl->tile_bytes = default_head_tile_bytes(s, d, kHeadTileTarget);
}

// A plan that only ever copies whole blocks between two head-major pools with the same head
// partition and block size moves each block as one span of identical bytes: it is copied as a
// contiguous plan. False (plan unchanged) for any other pair of layouts.
bool as_whole_block_copy(kvx_plan_s *pl) {
    const Geom &s = pl->src, &d = pl->dst;
    if (s.layout != KVX_LAYOUT_HND || d.layout != KVX_LAYOUT_HND || s.n_shards != d.n_shards ||
        s.heads_per_shard != d.heads_per_shard || s.block_size != d.block_size)
        return false;
    pl->per_head = 0;
    pl->strided = 0;
    pl->width = (int32_t)s.row_bytes();
    pl->src_pitch = s.row_bytes();
    pl->dst_pitch = d.row_bytes();
    pl->src_head_pitch = 0;
    pl->dst_head_pitch = 0;
    pl->tile_bytes = default_tile_bytes(s, d);
    return true;
}

// Bulk copies need 16-byte aligned addresses, sizes, widths and pitches (vec == 16), a ring that
// fits shared memory and, for strided plans, a row that fits a stage. The automatic choice, measured
// on GB300: a layer push that reads under 128 MiB runs fastest with the bulk kernel at two CTAs per
// SM (it leaves room for the caller's compute and the next push), a larger one with the persistent
// kernel at 128 threads per CTA and the occupancy limit of CTAs (many small independent CTAs). Plans
// that map one head layout onto another (head-group tiles: dozens of row copies per tile, too many for
// one issuing thread) take tensor-map copies (one TMA operation per tile and side) at any size, or
// the persistent kernel at 128 threads per CTA where no tensor map fits. Two head-major sides alike
// copy whole blocks as single spans and keep the bulk kernel (0.94-0.95 against 0.76).
constexpr int64_t kLargeLayer = (int64_t)128 << 20;

// The box of a TENSOR plan's maps: tiles of box_n token slots for box_k heads go through the maps
// (segments of min(block sizes) tokens, or tile_bytes / head_bytes of them when a head's segment is
// longer than a tile; as many heads as build_head_tiles puts in such a tile).
// The box order is the layout of the box in shared memory. A side whose layout is the box order and
// whose box is one contiguous span (token-major: all of a shard's heads; head-major: all of a block's
// slots) moves a box by one plain bulk copy, and only the other side through its map, which then does
// the transpose. The consumer side is preferred (measured on GB300, 32 MiB per layer in the per-layer
// step: head-major -> token-major 0.870 with maps on both sides against 0.917 with a plain store,
// token-major -> head-major 0.871 against 0.893 with a plain load; the tensor-map load transposes
// faster than the store).
bool tensor_side_flat(const Geom &g, int32_t order, int32_t box_n, int32_t box_k) {
    return g.layout == order && (order == KVX_LAYOUT_NHD ? box_k == g.heads_per_shard : box_n == g.block_size);
}

static void tensor_box(kvx_plan_s *pl) {
    const int64_t hb = pl->src.head_bytes();
    const int64_t rows = std::max<int64_t>(1, pl->tile_bytes / hb);
    const int64_t seg = std::min(pl->src.block_size, pl->dst.block_size);
    const int32_t group = std::min(pl->src.heads_per_shard, pl->dst.heads_per_shard);
    pl->box_n = (int32_t)std::min<int64_t>(seg, rows);
    pl->box_k = pl->box_n == seg ? (int32_t)std::min<int64_t>(group, std::max<int64_t>(1, rows / seg)) : 1;
    if (tensor_side_flat(pl->dst, pl->dst.layout, pl->box_n, pl->box_k))
        pl->box_order = pl->dst.layout;
    else if (tensor_side_flat(pl->src, pl->src.layout, pl->box_n, pl->box_k))
        pl->box_order = pl->src.layout;
    else
        pl->box_order = KVX_LAYOUT_NHD;
}

// A TENSOR plan needs head rows the maps can describe (16..2048 bytes, 16-byte multiples, a box of
// at most 256 per dimension that fits a ring stage) and host-built tiles.
static bool tensor_ok(const kvx_plan_s *pl) {
    const int64_t hb = pl->src.head_bytes();
    return pl->per_head && !same_head_major(pl->src, pl->dst) && !pl->device_built && pl->vec == 16 && hb % 16 == 0 &&
           hb <= 2048 && pl->box_n >= 1 && pl->box_n <= 256 && pl->box_k >= 1 && pl->box_k <= 256 &&
           (int64_t)pl->box_n * pl->box_k * hb <= pl->tile_bytes &&
           (int64_t)align_up((size_t)pl->tile_bytes, 128) * pl->bulk_stages <= kBulkRingMax;
}

static void resolve_kernel(kvx_plan_s *pl) {
    const bool bulk_ok = pl->vec == 16 && (int64_t)pl->tile_bytes * pl->bulk_stages <= kBulkRingMax &&
                         (!pl->strided || pl->width <= pl->tile_bytes);
    // STAGED: strided tiles whose rows are whole 16-byte vectors (loads by the bulk engine, stores by
    // the CTA's threads)
    const bool staged_ok = bulk_ok && pl->strided && pl->width % 16 == 0;
    const bool large = pl->bytes_per_layer >= kLargeLayer;
    const bool automatic = pl->kernel == KVX_KERNEL_AUTO;
    const bool row_groups = pl->per_head && !same_head_major(pl->src, pl->dst);
    tensor_box(pl);
    int32_t k = pl->kernel;
    // plans that map one head layout onto another: tensor-map copies (measured on GB300, 32 MiB per
    // layer: 0.95-0.96 of the copy peak in the per-layer step against 0.81 for PERSIST and 0.83-0.90
    // for STAGED; one 497 MB layer of the batched workload 1.00 against 0.968 for PERSIST, 0.87 for
    // STAGED), in a 2-stage ring for tiles above 16 KiB, else 4 stages (3 where 4 do not fit)
    if ((automatic || pl->kernel == KVX_KERNEL_TENSOR) && row_groups && tensor_ok(pl) && !pl->bulk_stages_req) {
        pl->bulk_stages = pl->tile_bytes > kHeadTileTarget ? 2 : 4;
        if (!tensor_ok(pl)) pl->bulk_stages = 3;
    }
    if (automatic) k = row_groups ? (tensor_ok(pl) ? KVX_KERNEL_TENSOR : KVX_KERNEL_PERSIST)
                                  : (bulk_ok && !large ? KVX_KERNEL_BULK : KVX_KERNEL_PERSIST);
    if (k == KVX_KERNEL_TENSOR && !tensor_ok(pl)) k = row_groups ? KVX_KERNEL_PERSIST : KVX_KERNEL_BULK;
    if (k == KVX_KERNEL_STAGED && !staged_ok) k = bulk_ok ? KVX_KERNEL_BULK : KVX_KERNEL_PERSIST;
    if (k == KVX_KERNEL_BULK && !bulk_ok) k = KVX_KERNEL_PERSIST;
    pl->kernel = k;
    pl->threads = pl->threads_req ? pl->threads_req : (automatic && (large || row_groups) ? 128 : 256);
}

// Default ring depth: 3 stages (measured on GB300: strided tiles, rows scattered on one side, ran
// fastest with 3; contiguous ones at 2 CTAs per SM with 3 stages reached 0.999 of the copy peak in
// the per-layer step and 0.81 for a launch alone, against 0.991 / 0.81 with 4 stages at 1.25 CTAs
// per SM).
static void resolve_stages(kvx_plan_s *pl) {
    pl->bulk_stages = pl->bulk_stages_req ? pl->bulk_stages_req : 3;
}

void resolve_launch(kvx_plan_s *pl) {
    resolve_stages(pl);
    resolve_kernel(pl);
}

void finish_plan_shape(kvx_plan_s *pl) {
    pl->vec = vector_bytes(pl, shard_pairs(pl->src, pl->dst));
    int64_t toks = pl->device_built ? pl->device_tokens : 0;
    for (int32_t n : pl->run_ntok) toks += n;
    pl->bytes_per_layer = toks * pl->src.row_bytes() * pl->src.n_shards * pl->src.n_planes;
    const int32_t kernel_req = pl->kernel;   // as asked (resolve_kernel replaces it with the resolved one)
    resolve_stages(pl);
    resolve_kernel(pl);
    // a TENSOR plan whose tile is the library's takes the larger TENSOR tile (its tiles are built
    // after this), unless that tile no longer resolves to TENSOR
    if (pl->kernel == KVX_KERNEL_TENSOR && pl->head_tile_auto && !pl->device_built) {
        const int32_t small = pl->tile_bytes;
        pl->tile_bytes = default_head_tile_bytes(pl->src, pl->dst, kTensorTileTarget);
        pl->kernel = kernel_req;
        resolve_stages(pl);
        resolve_kernel(pl);
        if (pl->kernel != KVX_KERNEL_TENSOR) {
            pl->tile_bytes = small;
            pl->kernel = kernel_req;
            resolve_stages(pl);
            resolve_kernel(pl);
        }
    }
}

}  // namespace kvx
