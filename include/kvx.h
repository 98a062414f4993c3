/*
 * kvx -- paged KV-cache push between two pools resident in one GPU's HBM (sm_103a).
 *
 * The calls below restate, for a single-GPU C library, the data path of the KV connectors described
 * in three web pages on disaggregated prefill/decode serving:
 *   [P1] the push-mode NIXL connector article (spke.com, article 3844);
 *   [P2] the "vLLM MoRIIO KV Connector" notes (single-node PD disaggregation);
 *   [P3] the bidirectional KV transfer article (spke.com, article 3845).
 * Section names are the pages' own.
 *
 * Conventions shared by every call:
 *  - Device memory (pools, token and id arrays given as device pointers) belongs to the caller.
 *    kvx allocates device memory only for plan descriptors, hash tables and the scratch of
 *    kvx_match_prefix / kvx_block_hashes, and frees it in kvx_plan_destroy / kvx_table_destroy or
 *    before the call returns.
 *  - Host arrays passed in are copied before the call returns; the caller may reuse them.
 *  - Every call returns a kvx_status. On error a one-line reason is stored in a thread-local
 *    buffer (kvx_last_error); no call aborts the process or traps on the device.
 *  - A plan or table is used by one host thread at a time. Different plans are independent.
 *  - Device work runs on the stream the caller passes (plus a library-owned non-blocking stream
 *    for small status read-backs).
 *  - The library keeps per-device state for the life of the process: its push lanes (streams), a
 *    stream-ordered memory pool, an event pool, the read-back stream and the device address of the
 *    fixed scratch of kvx_match_prefix_static. All of it belongs to the device's primary context:
 *    resetting the device (cudaDeviceReset) or otherwise destroying that context while the library
 *    is loaded leaves it dangling, and later calls on that device are undefined.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvx_status {
    KVX_OK = 0,
    KVX_EINVAL = 1,        /* malformed argument: null pointer, bad geometry, overlapping buffers  */
    KVX_ERANGE = 2,        /* block id outside [0, n_blocks) or too few ids for n_tokens          */
    KVX_EOVERLAP = 3,      /* a consumer block would be written by two requests (or twice)        */
    KVX_EUNSUPPORTED = 4,  /* layout pair the library does not map (shard counts do not divide)   */
    KVX_ENOMEM = 5,        /* device or host allocation failed; free list too short               */
    KVX_ECUDA = 6,         /* a CUDA runtime call failed (text in kvx_last_error)                 */
    KVX_ETIMEDOUT = 7,     /* kvx_sync deadline passed with pushes still pending                  */
    KVX_EFAILED = 8        /* a completed push reported FAILED for at least one layer             */
} kvx_status;

/* Per-layer state of a plan's pushes, [P2] section 6 ("failure handling": the batch state is decided
 * over all layers' states DONE / FAILED / PENDING, because a middle layer can fail). */
typedef enum kvx_layer_state {
    KVX_LAYER_IDLE = 0,     /* not pushed since the plan was built */
    KVX_LAYER_PENDING = 1,
    KVX_LAYER_DONE = 2,
    KVX_LAYER_FAILED = 3
} kvx_layer_state;

/*
 * One side's paged KV pool. [P2] section 3 (the one-time handshake exchanges the KV base address,
 * block size and per-layer tensor strides a peer needs to address the cache) and section 6
 * ("memory registration": each layer's KV tensor is registered separately).
 *
 * The pool is n_layers * n_planes * n_shards separate device buffers; buffer
 * base[(layer * n_planes + plane) * n_shards + shard] is a dense row-major array
 *     [n_blocks][block_size][heads_per_shard][head_dim]  (layout KVX_LAYOUT_NHD), or
 *     [n_blocks][heads_per_shard][block_size][head_dim]  (layout KVX_LAYOUT_HND)
 * of elem_bytes-byte elements. The two sides may use different layouts.
 * planes: 2 for separate K and V, 1 for a single latent (MLA). Shard s holds the global KV heads
 * [s * heads_per_shard, (s + 1) * heads_per_shard), i.e. the tensor-parallel head partition.
 * Values are moved as opaque bytes; elem_bytes only sizes them. `base` is a host array of buffer
 * pointers, copied by kvx_plan. Buffers are normally device memory; a pool may also live in pinned
 * host memory (or pageable host memory where the GPU can reach it), which the copy kernels reach over
 * the chip-to-chip link with plain loads and stores (the bulk copy path is kept to device memory;
 * the first push checks the first and last buffer of each pool, and a pool's buffers are expected
 * to be of one kind).
 */
#define KVX_LAYOUT_NHD 0
#define KVX_LAYOUT_HND 1

typedef struct kvx_pool {
    int32_t n_layers;
    int32_t n_planes;
    int32_t n_shards;
    int32_t heads_per_shard;
    int32_t head_dim;
    int32_t elem_bytes;
    int32_t block_size;     /* tokens per block */
    int32_t layout;         /* KVX_LAYOUT_NHD (0) or KVX_LAYOUT_HND (1) */
    int64_t n_blocks;
    void *const *base;
} kvx_pool;

/*
 * One request: its first n_tokens tokens are copied. Token t lives in producer block
 * src_block_ids[t / src.block_size] slot t % src.block_size, and goes to consumer block
 * dst_block_ids[t / dst.block_size] slot t % dst.block_size ([P1] "Implementierungsdetails",
 * step 3: each side maps block positions to its own physical layout, so block sizes may differ).
 * Unused slots of a last, partial consumer block keep their bytes. Host arrays.
 */
typedef struct kvx_request {
    int64_t req_id;
    int64_t n_tokens;
    const int32_t *src_block_ids;
    int32_t n_src;           /* >= ceil(n_tokens / src.block_size); extra ids are ignored */
    const int32_t *dst_block_ids;
    int32_t n_dst;           /* >= ceil(n_tokens / dst.block_size); extra ids are ignored */
} kvx_request;

typedef struct kvx_plan_s *kvx_plan_t;

/* Tuning knobs of a plan; zero fields take the defaults. */
typedef struct kvx_plan_opts {
    int32_t tile_bytes;       /* bytes one CTA copies per tile (multiple of 16). Default: 16384 for
                                 strided plans; for contiguous ones the block-row unit
                                 (min block size x row bytes) split into the fewest equal tiles
                                 of at most 16384 bytes, or whole units packed up to 16384     */
    int32_t threads;          /* threads per CTA of TILE / PERSIST (multiple of 32, <= 1024;
                                 default 256, or 128 where AUTO picks PERSIST for a large push
                                 or a head-group plan; BULK and TENSOR run 32, STAGED 128) */
    int32_t flags;            /* KVX_PLAN_* bits                                                 */
    int32_t kernel;           /* KVX_KERNEL_*; 0 lets the library choose                         */
    int32_t ctas_per_sm;      /* persistent kernels: resident CTAs per SM, capped at the occupancy
                                 limit (0: for launches that read under 128 MiB 2 per SM with the
                                 ring kernels (BULK, TENSOR, STAGED) and with PERSIST (4 for
                                 head-group tiles), leaving room for the caller's compute and an
                                 overlapping push; the occupancy limit for larger launches) */
    int32_t lanes;            /* internal streams pushes fan out over (0: the default, 1: none):
                                 4, or half the hardware work queues of the process
                                 (CUDA_DEVICE_MAX_CONNECTIONS, 8 when unset) when that is fewer,
                                 at least 1. Streams beyond the queues share them, and a lane that
                                 shares a queue with the caller's compute stream waits behind it:
                                 run with CUDA_DEVICE_MAX_CONNECTIONS >= 2 x (lanes + the caller's
                                 own streams) so that pushes overlap as intended                 */
    int32_t bulk_stages;      /* ring kernels: shared-memory stages of tile_bytes each, one of 2, 3,
                                 4, 6, 8 with stages * tile_bytes <= 192 KiB (0: 3; 4 for TENSOR
                                 chosen by AUTO)                                                 */
    int32_t layers_per_launch; /* kvx_push_layers: layers one copy launch covers, the launches of a
                                 call spread over the lanes (0: as many as make about 256 MiB
                                 moved, read + write, per launch when lanes > 1, at least one;
                                 the whole range in one launch when lanes = 1)                   */
    int32_t max_ctas;         /* upper bound on the CTAs of one copy launch (0: none). A push beside
                                 a kernel that fills whole SMs -- a tensor-core GEMM holding every
                                 register of an SM -- costs that kernel the SMs the copy occupies;
                                 a few CTAs with a deep ring (bulk_stages) move the same bytes on
                                 fewer SMs for longer                                            */
} kvx_plan_opts;

/* STAGED (strided plans with rows of whole 16-byte vectors): the bulk ring with 128 threads per
 * CTA. A tile lands in its stage in the producer's row order (one bulk copy when the producer side
 * of the tile is one span, else one per token or per row); the threads then store every row to its
 * place in the consumer's layout with 16-byte stores, so a head transpose needs no ring slot on the
 * store side.
 * TENSOR (plans with one token-major and one head-major side, or head-major sides that differ in
 * block size or head split): the bulk ring of BULK, but each tile of a head group is one box of a
 * tensor map (TMA). Every pool buffer gets a map over its own layout's strides, with the box laid
 * out in shared memory in one layout for both sides (the consumer's when a box is one contiguous
 * span of the consumer, else the producer's when it is one of the producer's, else token-major). A
 * side that holds the box as one span in that layout moves it with one plain bulk copy; the other
 * side moves it with one tensor-map load or store, which does the transpose. Default tiles: the most
 * shared heads of one block segment that fit 32 KiB, in a 2-stage ring. Tiles of another shape (a
 * partial last block) move row by row. Needs 16-byte aligned buffers and head rows of 16..2048 bytes
 * in multiples of 16; host-built plans only; otherwise PERSIST. */

/* Copy kernels. TILE: one CTA per tile. PERSIST: a grid of (SMs x resident CTAs) walks the tiles,
 * loading the next descriptor while it copies the current tile. BULK: the same walk with the bulk
 * asynchronous copy engine (global -> shared -> global through a ring of mbarrier-tracked stages;
 * strided tiles move row by row on a side whose rows are not adjacent); plans whose buffer bases,
 * offsets, widths and pitches are all 16-byte aligned, with a row no larger than tile_bytes; others
 * fall back to PERSIST. Contiguous BULK launches that read at least 8 MiB mark the lines they touch
 * evict-first in L2 (a cache hint only; the bytes copied are the same). AUTO picks BULK where it
 * applies to a plan that reads under 128 MiB per layer (two CTAs per SM with a 3-stage ring, leaving
 * room for the caller's compute and the next push) and PERSIST with 128 threads per CTA otherwise
 * (measured fastest on GB300 for large layer pushes); plans with one token-major and one head-major
 * side, or two head-major sides with different block sizes or head splits, take TENSOR (32 KiB
 * tiles, 2-stage ring) at any size when the tensor maps can describe them, else PERSIST. */
#define KVX_KERNEL_AUTO 0
#define KVX_KERNEL_TILE 1
#define KVX_KERNEL_PERSIST 2
#define KVX_KERNEL_BULK 3
#define KVX_KERNEL_TENSOR 4
#define KVX_KERNEL_STAGED 5

/* Record when every push starts and ends on the device; read with kvx_plan_push_times after
 * kvx_sync. The copy kernels stamp the GPU's global timer themselves (the first CTA to start, the
 * last CTA to finish), so timing adds no host call to a push. This is the per-layer KV transfer time
 * that the bidirectional article's prefill-duration breakdown ([P3] "Leistungsdaten", Figs. 4 and 6)
 * separates from recompute time. Up to 4096 pushes between two syncs are timed. */
#define KVX_PLAN_TIMING 1

/*
 * kvx_plan -- build the copy plan of a set of requests.
 * [P1] "Threading-Modell": the block ids of a request are mapped to memory descriptors and
 * contiguous blocks are merged into larger transfer regions; [P2] section 6 ("memory registration
 * and offset calculation"): transfers are (local offset, remote offset, size) triples and adjacent
 * blocks merge; [P2] section 6 ("rank mapping"): the two sides may use different TP sizes when one
 * is a multiple of the other.
 *
 * Runs are merged within each request at token granularity: a run is a maximal token range whose
 * producer rows (block * block_size + slot) and consumer rows both advance by one per token. Runs
 * are then cut into tiles of about tile_bytes for the copy kernel. The plan is layer-invariant:
 * a push for layer l only changes the buffer bases.
 *
 * Validation, all before any CUDA call (so kvx_plan runs without a GPU):
 *   EINVAL        null pointers, counts < 1, n_layers / n_planes / head_dim / elem_bytes differ,
 *                 total heads differ, null buffer, a consumer buffer overlaps any other buffer;
 *   EUNSUPPORTED  neither shard count divides the other; more than 2^31-1 rows in a buffer;
 *                 an unknown layout;
 *   ERANGE        a needed block id is outside [0, n_blocks), n_src or n_dst too small;
 *   EOVERLAP      a consumer block appears twice among all requests' needed ids.
 * No device memory is touched by kvx_plan; descriptors go to the device at the first push.
 * `opts` may be NULL.
 */
kvx_status kvx_plan(const kvx_pool *src, const kvx_pool *dst, const kvx_request *reqs, int32_t n_reqs,
                    kvx_plan_t *out);
kvx_status kvx_plan_ex(const kvx_pool *src, const kvx_pool *dst, const kvx_request *reqs, int32_t n_reqs,
                       const kvx_plan_opts *opts, kvx_plan_t *out);

/* Changes a plan's launch options before or between pushes (no push pending): flags, kernel,
 * threads, ctas_per_sm and lanes. tile_bytes must be 0 or the plan's own (its tiles are built).
 * Useful for plans built by kvx_match_prefix, which takes no options. */
kvx_status kvx_plan_set_opts(kvx_plan_t plan, const kvx_plan_opts *opts);

/* Introspection for tests: the plan's merged token runs (host arrays owned by the plan, valid
 * until kvx_plan_destroy). Rows are block * block_size + slot on each side. A plan built by
 * kvx_match_prefix keeps its runs on the device (no push needs them on the host); the first call
 * here copies them back with a synchronous copy. */
kvx_status kvx_plan_runs(kvx_plan_t plan, int64_t *n_runs, const int32_t **src_row,
                         const int32_t **dst_row, const int32_t **n_tokens);

/* Plan summary: runs, tiles per (layer, plane), bytes moved per layer (read; the same is written),
 * the vector width the copy kernel uses (16, 8, 4, 2 or 1 bytes), and whether rows are strided
 * (head-shard remap: each tile copies `n` rows of `width` bytes, stepping by the producer and
 * consumer row sizes) or contiguous (each tile copies `n` bytes). */
typedef struct kvx_plan_info {
    int64_t n_runs;
    int64_t n_tiles;             /* per (layer, plane) */
    int64_t bytes_per_layer;     /* read per layer; the same amount is written */
    int32_t vec_bytes;
    int32_t strided;
    int32_t n_layers;
    int32_t n_planes;
    int32_t width;               /* strided plans: bytes per row segment */
    int32_t tile_bytes;
    int32_t kernel;              /* the KVX_KERNEL_* the pushes use */
    int32_t threads;
    int32_t lanes;
    int32_t bulk_stages;         /* ring stages of the BULK kernel; 0 for the others */
    int64_t src_pitch;           /* strided plans: bytes between consecutive rows of a tile, producer */
    int64_t dst_pitch;           /* and consumer side */
    int64_t src_head_pitch;      /* plans with a head-major side: bytes between consecutive heads of a */
    int64_t dst_head_pitch;      /* tile (tiles then cover `heads` heads of n rows each), producer and consumer */
} kvx_plan_info;
kvx_status kvx_plan_get_info(kvx_plan_t plan, kvx_plan_info *out);

/* Introspection for tests: the tile table of a host-built plan (host memory owned by the plan).
 * Entry layout, 32 bytes: { int64 src_off; int64 dst_off; int32 n; int32 src_shard;
 * int32 dst_shard; int32 heads }; strided tiles copy n rows for each of max(heads, 1) heads. Offsets are bytes into the (layer, plane, shard) buffers; every
 * layer and plane uses the same table. Device-built plans report 0 entries here. */
kvx_status kvx_plan_tiles(kvx_plan_t plan, int64_t *n_tiles, const void **tiles);

/*
 * kvx_push_layer -- copy layer `layer` of every request of the plan, on `stream`.
 * [P2] section 3.2 (WRITE mode): after each layer's forward step the write of that layer is queued
 * to a worker that first synchronises on a CUDA event, so the copy of layer k starts after layer k's
 * compute and overlaps layer k+1; [P1] "Threading-Modell": the main loop hands the blocks to a
 * background thread and returns to model execution at once.
 *
 * The push is ordered after everything already enqueued on `stream` and, if `ready` is not NULL,
 * after `ready`. The call only enqueues: it returns before the copy runs. Completion is what
 * kvx_sync reports, not stream order: with lanes > 1 (the default) the copy runs on one of the
 * library's internal high-priority streams ("lanes", forked from `stream` by an event), so
 * consecutive pushes of different layers can overlap on the GPU, the head of one hiding the tail
 * of the previous; work enqueued on `stream` later is not ordered after the copy. Lanes run at the
 * priority of `stream`, so the caller decides whether pushes yield to its compute. With lanes = 1
 * the copy is enqueued on `stream` itself. Until kvx_sync returns KVX_OK the producer layer must
 * not be rewritten and the consumer layer must not be read. The first push of a plan allocates and
 * uploads its descriptors on `stream`. The current device must be the device of the pools and the
 * stream.
 * kvx_push_layers does layers [layer_begin, layer_end): with lanes > 1 in launches of
 * layers_per_launch layers each, on successive lanes, every one ordered after `stream` and `ready`
 * (measured on GB300: one launch for 64 layers of a 496 MB-per-layer batch reached 0.96-0.99 of the
 * copy peak, launches of about 256 MiB or one layer each 1.02-1.03, the heads of later launches
 * filling the tails of earlier ones); with lanes = 1 on `stream`, in one launch unless
 * layers_per_launch asks for more.
 */
kvx_status kvx_push_layer(kvx_plan_t plan, int32_t layer, cudaStream_t stream, cudaEvent_t ready);
kvx_status kvx_push_layers(kvx_plan_t plan, int32_t layer_begin, int32_t layer_end, cudaStream_t stream,
                           cudaEvent_t ready);

/* The same, and `done` (the caller's event, not NULL) is recorded right after the copy, on the
 * stream that runs it (after every launch of a multi-layer push, the last one's lane first waiting
 * for the others): a per-push completion notification ([P1] "Implementierungsdetails", step 3:
 * each write carries a completion notification). A consumer stream can wait on it before reading
 * the layer; kvx_sync still reports failures. */
kvx_status kvx_push_layer_notify(kvx_plan_t plan, int32_t layer_begin, int32_t layer_end, cudaStream_t stream,
                                 cudaEvent_t ready, cudaEvent_t done);

/*
 * kvx_sync -- wait for every push issued on the plan since the last completed sync.
 * [P1] "Implementierungsdetails", step 3: the consumer counts one completion per producer write and
 * treats the KV as received only when all expected completions arrived; [P2] section 3.2
 * (wait_for_save seals the number of writes actually queued) and section 6 (per-layer batch state).
 *
 * The count is sealed at entry: pushes issued so far. timeout_us < 0 waits without a deadline;
 * otherwise the host polls until the deadline and returns KVX_ETIMEDOUT with the pushes still
 * pending (a later kvx_sync waits for them again). When all are complete: KVX_EFAILED if any layer
 * reported FAILED (kvx_plan_layer_states tells which), else KVX_OK.
 */
kvx_status kvx_sync(kvx_plan_t plan, int64_t timeout_us);

/* Plans built with KVX_PLAN_TIMING: for each push the last completed kvx_sync confirmed, in issue
 * order, its start and end in microseconds relative to the earliest start among them (up to cap
 * entries each; *n receives the count). A push starts when the first CTA of its kernel starts and
 * ends when the last one has finished (its stores completed). Pushes on different lanes may overlap.
 * A push with nothing to copy launches no kernel and has no entry. */
kvx_status kvx_plan_push_times(kvx_plan_t plan, float *start_us, float *end_us, int32_t cap, int32_t *n);

/* The same entries as raw readings of the GPU's global timer (nanoseconds). One clock serves the
 * whole device, so the pushes of different plans can be placed on one timeline. */
kvx_status kvx_plan_push_times_ns(kvx_plan_t plan, int64_t *start_ns, int64_t *end_ns, int32_t cap, int32_t *n);

/* Per-layer states (out: n_layers entries of kvx_layer_state). */
kvx_status kvx_plan_layer_states(kvx_plan_t plan, int32_t *out, int32_t n_layers);

/* Testing hook for host-side fault injection: the next push of `layer` completes normally on the
 * device but is reported FAILED by kvx_sync. */
kvx_status kvx_plan_inject_failure(kvx_plan_t plan, int32_t layer);

/* Testing hook for the copy kernel's bounded device-side wait ([P2] section 3.1: failed loads are
 * reported and those blocks recomputed; section 6: a middle layer can fail). The next push of
 * `layer` runs with a 1 ms limit on each wait for a bulk ring stage instead of 2 s, and the
 * launch's first CTA, once the loads of its first work item of that layer have landed, waits for a
 * phase of that stage that nothing arms: a wait that can only run out, with no copy in flight. The
 * CTA gives up at the limit, marks every layer of the work it had left FAILED, waits (at most the
 * limit each) for its loads still in flight and returns; the other CTAs finish normally and nothing
 * faults. kvx_sync then reports KVX_EFAILED and the layer
 * FAILED; consumer bytes the CTA did not copy keep their prior contents. KVX_EUNSUPPORTED unless the
 * plan's pushes run the bulk kernel. */
kvx_status kvx_plan_inject_stall(kvx_plan_t plan, int32_t layer);

/* Waits for any pending push, then frees the plan and its device descriptors. NULL is a no-op.
 * kvx_sync and kvx_plan_destroy make the plan's device (current at its first push, or at
 * kvx_match_prefix for a device-built plan) current while they run and restore the caller's;
 * kvx_table_destroy does the same with the device current at kvx_table_build. */
kvx_status kvx_plan_destroy(kvx_plan_t plan);

const char *kvx_status_str(kvx_status status);
const char *kvx_last_error(void);

/* ------------------------------------------------------------------------------------------------
 * Bidirectional reuse: block hashes, local prefix table, match and decode->prefill plan.
 * [P3] "Bidirektionaler KV-Transfer", Figure 1 steps 4-6: prefill checks the remote reusable KV
 * after applying local cache hits, queues a receive when the reusable tokens reach the threshold,
 * and the same transfer mechanism moves the blocks decode->prefill; [P3] "KV-Recompute-
 * Schwellenwert": recompute below kv_recompute_threshold, pull at or above it.
 * ---------------------------------------------------------------------------------------------- */

/*
 * kvx_block_hashes -- chained block hashes of sessions' token streams, on `stream` (waits for it).
 * Session s has tokens[tok_off[s] .. tok_off[s+1]) (uint32 ids, device CSR; tok_off is a device
 * array of n_sessions + 1 int64). For each full block j (block_size tokens), the hash is 64-bit
 * FNV-1a (offset basis 14695981039346656037, prime 1099511628211; per octet xor then multiply)
 * over the parent hash as 8 little-endian octets followed by the block's token ids as 4
 * little-endian octets each; block 0's parent is 0. A trailing partial block is not hashed.
 * Output for session s goes to out_hash[hash_off[s] ...] (device; hash_off device, n_sessions + 1
 * int64, each session needing floor(len / block_size) slots). The pages name prefix caching but
 * not the hash; this chained FNV-1a is the reading this library fixes.
 */
kvx_status kvx_block_hashes(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                            int32_t block_size, uint64_t *out_hash, const int64_t *hash_off,
                            cudaStream_t stream);

/* The same, continuing each session's chain: session s's first block chains to parent[s] (device
 * array of n_sessions uint64; NULL means 0 for every session, which is kvx_block_hashes). A session's
 * tokens then start at a block boundary of its whole stream and parent[s] is the hash of the block
 * before them, so a turn's newly filled blocks are hashed without the blocks before them. */
kvx_status kvx_block_hashes_ex(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                               int32_t block_size, const uint64_t *parent, uint64_t *out_hash,
                               const int64_t *hash_off, cudaStream_t stream);

/* Device hash table of the prefill side's resident blocks: hash -> local block id. */
typedef struct kvx_table_s *kvx_table_t;

/* Builds a table from n device keys / values on `stream` and waits for it. Duplicate keys ->
 * KVX_EINVAL (no table). n may be 0. */
kvx_status kvx_table_build(const uint64_t *keys, const int32_t *vals, int64_t n, cudaStream_t stream,
                           kvx_table_t *out);
/* Looks up n device keys; out_vals[i] = value or -1 (device). */
kvx_status kvx_table_lookup(kvx_table_t table, const uint64_t *keys, int64_t n, int32_t *out_vals,
                            cudaStream_t stream);
/* Waits for the table's last lookup, then frees it. */
kvx_status kvx_table_destroy(kvx_table_t table);

/* Per-session decision of kvx_match_prefix (device array, one entry per session). */
typedef struct kvx_match_result {
    int32_t local_hit_blocks;   /* L_loc: longest prefix of blocks resident in the local table     */
    int32_t remote_hit_blocks;  /* L_rem: longest prefix whose hash equals the published hash      */
    int32_t missing_tokens;     /* max(0, L_rem - L_loc) * block_size                              */
    int32_t push;               /* 1 iff missing_tokens > 0 and missing_tokens >= threshold        */
    int64_t dst_start;          /* offset into free_blocks of the session's first block, or -1     */
} kvx_match_result;

/*
 * kvx_match_prefix -- decide, per session, whether to pull the decode-held span, and build the
 * decode->prefill plan.
 *
 * Inputs (device unless stated): tokens/tok_off as in kvx_block_hashes; the local table; the
 * published remote list per session, remote_hash/remote_blk[rem_off[s] .. rem_off[s+1]) (hash and
 * decode block id of each of the session's blocks, in order); recompute_threshold_tokens (host);
 * free_blocks[0 .. n_free) (distinct prefill blocks, handed out in order). Pushing sessions, in
 * session order, take (L_rem - L_loc) consecutive entries of free_blocks; pair k of session s
 * copies decode block remote_blk[rem_off[s] + L_loc + k] into prefill block
 * free_blocks[dst_start + k].
 *
 * remote_pool is the producer (decode) pool, local_pool the consumer (prefill) pool; their
 * block_size must equal block_size; their layouts and head partitions may differ as in kvx_plan
 * (whole blocks between head-major pools of the same partition move as identical byte spans, other
 * head-major pairs by groups of heads per block). If out_plan is not NULL it receives a plan (built on the
 * device) whose pushes copy those blocks with kvx_push_layer / kvx_sync; NULL computes the
 * decisions only (the pools may then be NULL). The call waits for `stream` (it reads back its
 * status; with a plan or hole filling also the published-block total first). Block ids outside a pool make the affected layers FAILED at kvx_sync (the copy kernel
 * skips them). If the pushing sessions need more than n_free blocks the decisions are still
 * written, no plan is made, and the call returns KVX_ENOMEM.
 */
kvx_status kvx_match_prefix(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                            int32_t block_size, kvx_table_t local_table, const uint64_t *remote_hash,
                            const int32_t *remote_blk, const int64_t *rem_off,
                            int32_t recompute_threshold_tokens, const int32_t *free_blocks, int64_t n_free,
                            const kvx_pool *remote_pool, const kvx_pool *local_pool, kvx_match_result *out,
                            kvx_plan_t *out_plan, cudaStream_t stream);

/*
 * Options of kvx_match_prefix_ex (all off when opts is NULL; kvx_match_prefix is that case).
 *  KVX_MATCH_FILL_HOLES: blocks of [0, L_rem) that are resident locally are reused even past the
 *    first local miss (a chained hash certifies a block's whole prefix); only the non-resident
 *    blocks of [0, L_rem) are pulled, in order: missing_tokens = their count * block_size.
 *  KVX_MATCH_KEEP_LAST: when the L_rem matching blocks cover every token of a session, the last of
 *    them is recomputed instead of pulled ([P2] section 3.1: the last token is always recomputed).
 *  expiry / now: retention of the published spans ([P3] "Block Retention TTL": a turn that arrives
 *    after the TTL falls back to normal prefill). expiry is a device array with one entry per
 *    session (any clock; now is on the same clock); a session with now >= expiry[s] has nothing
 *    published. NULL: spans never expire.
 */
#define KVX_MATCH_FILL_HOLES 1
#define KVX_MATCH_KEEP_LAST 2
/* Testing hook for the device-side bounded wait of the plan emission: the first tile of the
 * look-back scan that numbers the plan's runs publishes nothing and the scan's waits are bounded by
 * 1 ms, so the next tile's wait on it runs out (a scan of more than 1024 pulled blocks; nothing
 * faults). The call then returns KVX_ETIMEDOUT with no plan. */
#define KVX_MATCH_TEST_SCAN_STALL 256

typedef struct kvx_match_opts {
    int32_t flags;
    int32_t reserved0;             /* must be 0 */
    const int64_t *expiry;
    int64_t now;
    int64_t reserved[4];           /* must be 0 */
} kvx_match_opts;

kvx_status kvx_match_prefix_ex(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                               int32_t block_size, kvx_table_t local_table, const uint64_t *remote_hash,
                               const int32_t *remote_blk, const int64_t *rem_off,
                               int32_t recompute_threshold_tokens, const int32_t *free_blocks, int64_t n_free,
                               const kvx_pool *remote_pool, const kvx_pool *local_pool, const kvx_match_opts *opts,
                               kvx_match_result *out, kvx_plan_t *out_plan, cudaStream_t stream);

/*
 * kvx_match_prefix_static -- the per-session decision of kvx_match_prefix (the same
 * kvx_match_result per session, dst_start included) without allocating any memory. The pages have
 * no counterpart: this entry point exists for callers that cannot allocate device memory on the
 * request path, typically serving engines that reserve nearly all free HBM for their paged KV
 * pools at start-up, where a later cudaMalloc can fail and cudaMalloc / cudaFree may synchronise
 * the device and stall the other streams.
 *
 * Arguments as in kvx_match_prefix; no plan is built (free_blocks is not read, n_free only bounds
 * the assignment). Its scratch is one fixed array of the library (about 1 MiB on every GPU that
 * loads it, held until the process exits), sized for at most 65536 sessions per call; more
 * return KVX_EINVAL. The first call on a device looks up that array's device address and keeps it
 * for later calls (make this first call before any stream capture; a device reset invalidates it,
 * see the conventions at the top). Every call reuses the same array and leaves its contents
 * behind; the call clears what must start at zero. Calls whose device work overlaps (on different
 * streams or host threads) race on the array. The call waits for `stream`. Returns KVX_OK, or
 * KVX_ENOMEM with the decisions written when the pushing sessions need more than n_free blocks.
 */
kvx_status kvx_match_prefix_static(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                                   int32_t block_size, kvx_table_t local_table, const uint64_t *remote_hash,
                                   const int64_t *rem_off, int32_t recompute_threshold_tokens, int64_t n_free,
                                   kvx_match_result *out, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * Connector state machine (host only; no CUDA call, usable without a GPU).
 *
 * The protocol around the push, one record per request id:
 *   [P1] "Implementierungsdetails" step 1 (the consumer registers its destination blocks when it
 *        allocates them), step 2 (registration and end of prefill meet in either order; whichever
 *        comes second triggers the transfer; matching is by request id and copes with resent,
 *        preempted and retried requests) and step 3 (one completion per producer rank; the KV
 *        counts as received only when all expected completions are in);
 *   [P2] section 3.2 (a write task whose destination ids have not arrived waits on a deferred list
 *        and is given up after defer_timeout so the producer's blocks are freed; chunked prefill
 *        collects blocks until the last chunk; wait_for_save seals the number of writes actually
 *        queued), section 3.1 (failed loads are reported so those blocks are recomputed), section
 *        5 (transfer_timeout, defer_timeout, recv_abort_timeout) and section 6 (the batch state is
 *        decided over every layer's DONE / FAILED / PENDING; with consumer TP above producer TP,
 *        consumer_tp / producer_tp acknowledgements complete a request).
 *
 * States of a record (the attempt it belongs to is part of every event):
 *
 *   WAITING --register + last prefill chunk--> READY --kvx_conn_start--> IN_FLIGHT --all ranks
 *      |                                                                  sealed and reported-->
 *      +--last prefill chunk, no registration--> DEFERRED --register--> READY      DONE | FAILED
 *   DEFERRED --defer_timeout--> EXPIRED          IN_FLIGHT --transfer_timeout--> TIMED_OUT
 *   registered, not DONE/FAILED --recv_abort_timeout (from registration)--> ABORTED
 *
 * Time is the caller's: every call that can change a state takes `now_us` (any monotonic
 * microsecond clock; tests pass a fake one). Deadlines are checked by kvx_conn_poll only.
 * A call naming an attempt older than the record's is stale and ignored (KVX_OK, no change); a
 * newer attempt discards the record's state and starts over (a retried or preempted request).
 * kvx_conn_* calls may come from several host threads; one mutex per connector orders them.
 * Records stay until kvx_conn_release.
 * ---------------------------------------------------------------------------------------------- */
typedef struct kvx_conn_s *kvx_conn_t;

typedef enum kvx_conn_state {
    KVX_CONN_WAITING = 0,    /* nothing yet, or only the registration (held until prefill ends)  */
    KVX_CONN_DEFERRED = 1,   /* prefill done, no registration yet: the producer holds its blocks */
    KVX_CONN_READY = 2,      /* both halves in: the transfer may start                           */
    KVX_CONN_IN_FLIGHT = 3,
    KVX_CONN_DONE = 4,       /* every rank sealed and every write it queued reported, none failed */
    KVX_CONN_FAILED = 5,     /* as DONE, but a write reported a FAILED layer: see load errors     */
    KVX_CONN_EXPIRED = 6,    /* defer_timeout ran out while DEFERRED: free the producer's blocks  */
    KVX_CONN_TIMED_OUT = 7,  /* transfer_timeout ran out while IN_FLIGHT                          */
    KVX_CONN_ABORTED = 8     /* recv_abort_timeout ran out after registration                     */
} kvx_conn_state;

typedef struct kvx_conn_config {
    int64_t defer_timeout_us;      /* 0 selects 60 s  */
    int64_t transfer_timeout_us;   /* 0 selects 30 s  */
    int64_t recv_abort_timeout_us; /* 0 selects 120 s */
    int32_t n_ranks;               /* writer ranks (acknowledgements) that complete a request, at most
                                      65536; 0 selects 1 */
    int32_t reserved;              /* must be 0 */
} kvx_conn_config;

typedef struct kvx_conn_event {
    int64_t req_id;
    int32_t attempt;
    int32_t state;                 /* READY, DONE, FAILED, EXPIRED, TIMED_OUT or ABORTED */
} kvx_conn_event;

typedef struct kvx_conn_info {
    int32_t attempt;
    int32_t state;                 /* kvx_conn_state */
    int64_t n_tokens;              /* tokens the producer has computed (last kvx_conn_prefill) */
    int32_t n_src;                 /* producer block ids collected over all chunks so far */
    int32_t n_dst;                 /* registered consumer block ids */
    int32_t n_chunks;              /* prefill chunks received */
    int32_t ranks_sealed;
    int64_t writes_issued;         /* over all ranks */
    int64_t writes_expected;       /* over the sealed ranks */
    int64_t writes_done;           /* writes reported (failed ones included) */
    int64_t writes_failed;
    int32_t n_load_errors;         /* distinct consumer block ids to recompute */
    int32_t first_error;           /* position in the registered id list of the earliest failed block; -1 if none */
} kvx_conn_info;

/* cfg may be NULL (all defaults). KVX_EINVAL for negative values or reserved != 0. */
kvx_status kvx_conn_create(const kvx_conn_config *cfg, kvx_conn_t *out);
kvx_status kvx_conn_destroy(kvx_conn_t conn);   /* NULL is a no-op */

/* Consumer side: register the destination block ids (host array, copied). A resent registration
 * with the same ids is a no-op; with different ids, KVX_EINVAL. Completes the rendezvous (READY)
 * when the last prefill chunk is already in. KVX_ETIMEDOUT when this attempt already EXPIRED: the
 * producer gave up and the consumer must prefill the request itself. */
kvx_status kvx_conn_register(kvx_conn_t conn, int64_t req_id, int32_t attempt, const int32_t *dst_ids,
                             int32_t n_dst, int64_t now_us);

/* Producer side: one prefill chunk finished. Its block ids (host array, copied) are appended to the
 * request's; n_tokens is the request's computed length so far. Nothing can move before the last
 * chunk (last_chunk != 0): only then does the request become READY (registration in) or DEFERRED
 * (not yet). A chunk after the last one: KVX_EINVAL. */
kvx_status kvx_conn_prefill(kvx_conn_t conn, int64_t req_id, int32_t attempt, const int32_t *src_ids,
                            int32_t n_src, int64_t n_tokens, int32_t last_chunk, int64_t now_us);

/* Applies every deadline that has passed at now_us, then hands out up to cap pending events in the
 * order they happened (*n receives the count; the rest wait for the next poll). An event whose
 * record was released or restarted since is dropped. */
kvx_status kvx_conn_poll(kvx_conn_t conn, int64_t now_us, kvx_conn_event *out, int32_t cap, int32_t *n);

/* Snapshot of one record; KVX_EINVAL for an unknown id. */
kvx_status kvx_conn_get(kvx_conn_t conn, int64_t req_id, kvx_conn_info *out);

/* The producer (src) and consumer (dst) block ids of a record, for kvx_plan. KVX_ERANGE when a cap
 * is smaller than n_src / n_dst. */
kvx_status kvx_conn_ids(kvx_conn_t conn, int64_t req_id, int32_t *src, int32_t src_cap, int32_t *dst,
                        int32_t dst_cap);

/* READY -> IN_FLIGHT (the transfer_timeout clock starts). KVX_EINVAL from any other state. */
kvx_status kvx_conn_start(kvx_conn_t conn, int64_t req_id, int32_t attempt, int64_t now_us);

/* Producer rank `rank` (0 <= rank < n_ranks) queued n_writes more writes (pushes) for the request.
 * Only while IN_FLIGHT and before that rank sealed. */
kvx_status kvx_conn_write_issued(kvx_conn_t conn, int64_t req_id, int32_t attempt, int32_t rank,
                                 int32_t n_writes);

/* Rank `rank` queued all its writes: its expected count becomes the number it issued (a second
 * seal is a no-op). The request completes when every rank sealed and reported all its writes. */
kvx_status kvx_conn_seal(kvx_conn_t conn, int64_t req_id, int32_t attempt, int32_t rank);

/* One write of rank `rank` finished. layer_states: the per-layer states of the layers it covered
 * (kvx_layer_state, e.g. from kvx_plan_layer_states). All DONE: a good write. Any FAILED, even
 * among later DONE ones: a failed write, whose consumer blocks become load errors -- the
 * failed_blocks given (consumer ids), or every registered block when n_failed == 0. Any IDLE or
 * PENDING: KVX_EINVAL and nothing is counted. More reports than a sealed rank issued: KVX_EINVAL. */
kvx_status kvx_conn_write_done(kvx_conn_t conn, int64_t req_id, int32_t attempt, int32_t rank,
                               const int32_t *layer_states, int32_t n_layers, const int32_t *failed_blocks,
                               int32_t n_failed, int64_t now_us);

/* Consumer block ids whose KV did not arrive, in the order first reported (up to cap; *n receives
 * the full count). The consumer recomputes them. */
kvx_status kvx_conn_load_errors(kvx_conn_t conn, int64_t req_id, int32_t *blocks, int32_t cap, int32_t *n);

/* Forget a record (after its blocks were freed or handed to decode). Unknown ids are a no-op. */
kvx_status kvx_conn_release(kvx_conn_t conn, int64_t req_id);

/* Number of records held. */
int64_t kvx_conn_size(kvx_conn_t conn);

/* Library version string and the number of kvx kernels launched by this process so far. */
const char *kvx_version(void);
int64_t kvx_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KVX_H */
