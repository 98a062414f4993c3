/*
 * kvx oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the kvx hot path computes. Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg call it; the library never does, and the two
 * share no code, header, table or helper. Every function follows the loops of the definition it
 * cites, with no blocking, fusion or reordering.
 *
 * Sources (web pages on disaggregated prefill/decode KV transfer):
 *  [push]  "Push-based KV transfer" article (spke.com 3844), section "Implementierungsdetails",
 *          step 3 (transfer): the producer writes the KV blocks into the consumer's memory,
 *          addressing each target tensor-parallel rank; each side maps block positions to its own
 *          physical layout, so block sizes may differ between the sides.
 *  [runs]  same article, section "Threading-Modell": block ids are mapped to memory descriptors and
 *          contiguous blocks are merged into larger transfer regions; "vLLM MoRIIO KV Connector"
 *          notes, section 6 ("memory registration and offset calculation"): transfers are lists of
 *          (local offset, remote offset, size) triples and adjacent blocks are merged.
 *  [ranks] "vLLM MoRIIO KV Connector" notes, section 6 ("rank mapping"): prefill and decode may use
 *          different TP sizes when one is a multiple of the other.
 *  [match] "Bidirectional KV transfer" article (spke.com 3845), Figure 1 steps 4-6 (check the
 *          remote reusable KV after applying local cache hits; receive only when the reusable token
 *          count reaches the threshold) and section "KV-Recompute-Schwellenwert" (recompute below
 *          the threshold, pull at or above it).
 *  [fnv]   the FNV-1a hash as published by its authors (Fowler, Noll, Vo): 64-bit offset basis
 *          14695981039346656037, 64-bit prime 1099511628211; per octet: xor, then multiply.
 *
 * Readings where the pages are silent (all stated again in the design notes):
 *  - each (layer, plane, shard) buffer is dense [n_blocks][block_size][heads][head_dim] ("NHD"),
 *    or [n_blocks][heads][block_size][head_dim] ("HND") when the pool says so;
 *  - token t of a request lives in block ids[t / block_size], slot t % block_size, on each side;
 *  - only tokens [0, n_tokens) are copied, so unused slots of a last block keep their old bytes;
 *  - shard s owns the global heads [s*heads_per_shard, (s+1)*heads_per_shard);
 *  - runs merge within a request only;
 *  - a block hash is FNV-1a over the parent hash (8 bytes, little endian) then the block's token ids
 *    (4 bytes each, little endian); the first block's parent is 0; only full blocks are hashed;
 *  - missing = max(0, L_rem - L_loc) * block_size; push iff missing > 0 and missing >= threshold;
 *  - pushing sessions take prefill blocks from the free list in session order.
 * Options of the match (each off by default):
 *  - fill holes: blocks of [0, L_rem) that are resident locally are reused even past the first local
 *    miss (a chained hash certifies the whole prefix before the block), so only the non-resident
 *    blocks of [0, L_rem) are pulled: missing = that count * block_size;
 *  - TTL ("Bidirectional KV transfer" article, "Block Retention TTL": a turn arriving after the
 *    retention time falls back to normal prefill): a session whose published span has expiry <= now
 *    has nothing published;
 *  - keep last ("vLLM MoRIIO KV Connector" notes, section 3.1: the last token is always recomputed):
 *    when L_rem blocks cover every token of the session, L_rem drops by one block.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FNV64_OFFSET_BASIS 14695981039346656037ULL
#define ORACLE_FNV64_PRIME 1099511628211ULL

/* One side's pool, as the oracle sees it: host copies of each (layer, plane, shard) buffer. */
typedef struct {
    int32_t n_layers, n_planes, n_shards, heads_per_shard, head_dim, elem_bytes, block_size;
    int32_t layout; /* 0: [block][slot][head][dim], 1: [block][head][slot][dim] */
    int64_t n_blocks;
    uint8_t **base; /* [(layer * n_planes + plane) * n_shards + shard] */
} oracle_pool;

/* Index, in units of one head's bytes, of (block, slot, head) inside one buffer. */
static int64_t oracle_head_index(const oracle_pool *p, int64_t blk, int64_t slot, int64_t head)
{
    if (p->layout == 1) return (blk * p->heads_per_shard + head) * p->block_size + slot;
    return (blk * p->block_size + slot) * p->heads_per_shard + head;
}

/* ------------------------------------------------------------------------------------------- */
/* [push] [ranks]: the per-head byte copy, request -> layer -> plane -> token -> shard -> head.  */
/* Returns 0, or -1 if a block id is out of range or the head totals differ.                     */
/* ------------------------------------------------------------------------------------------- */
int oracle_push(const oracle_pool *src, const oracle_pool *dst, int32_t n_reqs,
                const int64_t *n_tokens, const int32_t *const *src_ids, const int32_t *const *dst_ids)
{
    if (src->n_shards * src->heads_per_shard != dst->n_shards * dst->heads_per_shard) return -1;
    if (src->head_dim * src->elem_bytes != dst->head_dim * dst->elem_bytes) return -1;
    const size_t head_bytes = (size_t)src->head_dim * (size_t)src->elem_bytes;
    for (int32_t r = 0; r < n_reqs; ++r) {
        for (int32_t l = 0; l < src->n_layers; ++l) {
            for (int32_t p = 0; p < src->n_planes; ++p) {
                for (int64_t t = 0; t < n_tokens[r]; ++t) {
                    int64_t sblk = src_ids[r][t / src->block_size];
                    int64_t dblk = dst_ids[r][t / dst->block_size];
                    if (sblk < 0 || sblk >= src->n_blocks || dblk < 0 || dblk >= dst->n_blocks) return -1;
                    int64_t src_slot = t % src->block_size;
                    int64_t dst_slot = t % dst->block_size;
                    for (int32_t s = 0; s < src->n_shards; ++s) {
                        for (int32_t h = 0; h < src->heads_per_shard; ++h) {
                            int32_t g = s * src->heads_per_shard + h;      /* global KV head */
                            int32_t ds = g / dst->heads_per_shard;         /* consumer shard */
                            int32_t dh = g % dst->heads_per_shard;         /* head within it */
                            const uint8_t *from = src->base[((int64_t)l * src->n_planes + p) * src->n_shards + s]
                                                  + (size_t)oracle_head_index(src, sblk, src_slot, h) * head_bytes;
                            uint8_t *to = dst->base[((int64_t)l * dst->n_planes + p) * dst->n_shards + ds]
                                          + (size_t)oracle_head_index(dst, dblk, dst_slot, dh) * head_bytes;
                            memcpy(to, from, head_bytes);
                        }
                    }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------- */
/* [runs]: maximal runs of one request's block list. A new run starts at block i when either    */
/* side's id is not its predecessor's id + 1. Returns the number of runs written.               */
/* ------------------------------------------------------------------------------------------- */
int32_t oracle_block_runs(int32_t n, const int32_t *src_ids, const int32_t *dst_ids,
                          int32_t *run_src, int32_t *run_dst, int32_t *run_len)
{
    int32_t nr = 0;
    for (int32_t i = 0; i < n; ++i) {
        int starts_run = (i == 0) || (src_ids[i] != src_ids[i - 1] + 1) || (dst_ids[i] != dst_ids[i - 1] + 1);
        if (starts_run) {
            run_src[nr] = src_ids[i];
            run_dst[nr] = dst_ids[i];
            run_len[nr] = 1;
            ++nr;
        } else {
            run_len[nr - 1] += 1;
        }
    }
    return nr;
}

/* Maximal runs at token granularity, for sides whose block sizes may differ: a new run starts at  */
/* token t when either side's row (block * block_size + slot) is not its predecessor's row + 1.   */
int64_t oracle_token_runs(int64_t n_tokens, int32_t bs_src, const int32_t *src_ids, int32_t bs_dst,
                          const int32_t *dst_ids, int64_t *run_src_row, int64_t *run_dst_row,
                          int64_t *run_len)
{
    int64_t nr = 0, prev_s = 0, prev_d = 0;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t srow = (int64_t)src_ids[t / bs_src] * bs_src + t % bs_src;
        int64_t drow = (int64_t)dst_ids[t / bs_dst] * bs_dst + t % bs_dst;
        if (t == 0 || srow != prev_s + 1 || drow != prev_d + 1) {
            run_src_row[nr] = srow;
            run_dst_row[nr] = drow;
            run_len[nr] = 1;
            ++nr;
        } else {
            run_len[nr - 1] += 1;
        }
        prev_s = srow;
        prev_d = drow;
    }
    return nr;
}

/* ------------------------------------------------------------------------------------------- */
/* [fnv]: FNV-1a over n octets, continuing from state h (pass the offset basis to start).       */
/* ------------------------------------------------------------------------------------------- */
uint64_t oracle_fnv1a64(const uint8_t *data, int64_t n, uint64_t h)
{
    for (int64_t i = 0; i < n; ++i) {
        h ^= (uint64_t)data[i];
        h *= ORACLE_FNV64_PRIME;
    }
    return h;
}

uint64_t oracle_fnv64_offset_basis(void) { return ORACLE_FNV64_OFFSET_BASIS; }

/* Chained block hashes of one token sequence: block j (full blocks only) hashes the octets of  */
/* its parent hash (8, little endian; parent of block 0 is 0) followed by its block_size token  */
/* ids (4 octets each, little endian). Returns the number of full blocks.                        */
int64_t oracle_block_hashes(const uint32_t *tokens, int64_t n_tokens, int32_t block_size, uint64_t *out)
{
    int64_t n_full = n_tokens / block_size;
    uint8_t *msg = (uint8_t *)malloc(8 + 4 * (size_t)block_size);
    if (!msg) return -1;
    uint64_t parent = 0;
    for (int64_t j = 0; j < n_full; ++j) {
        for (int b = 0; b < 8; ++b) msg[b] = (uint8_t)(parent >> (8 * b));
        for (int32_t i = 0; i < block_size; ++i) {
            uint32_t tok = tokens[j * block_size + i];
            for (int b = 0; b < 4; ++b) msg[8 + 4 * i + b] = (uint8_t)(tok >> (8 * b));
        }
        out[j] = oracle_fnv1a64(msg, 8 + 4 * (int64_t)block_size, ORACLE_FNV64_OFFSET_BASIS);
        parent = out[j];
    }
    free(msg);
    return n_full;
}

/* ------------------------------------------------------------------------------------------- */
/* [match]: the bidirectional reuse decision per session, then the decode->prefill block pairs. */
/* ------------------------------------------------------------------------------------------- */
static int oracle_cmp_u64(const void *a, const void *b)
{
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return (x > y) - (x < y);
}

static int oracle_is_resident(const uint64_t *sorted, int64_t n, uint64_t key)
{
    return bsearch(&key, sorted, (size_t)n, sizeof(uint64_t), oracle_cmp_u64) != NULL;
}

/*
 * Per session s (tokens[tok_off[s] .. tok_off[s+1]), published remote list
 * remote_hash/remote_blk[rem_off[s] .. rem_off[s+1])):
 *   h_j        = chained block hashes of the session's full blocks;
 *   L_loc      = longest prefix of blocks whose hashes are in local_keys (local cache hits);
 *   L_rem      = longest prefix of blocks whose hash equals the published remote hash at j;
 *   missing    = max(0, L_rem - L_loc) * block_size tokens;
 *   push       = missing > 0 and missing >= threshold.
 * Then, in session order, each pushing session takes (L_rem - L_loc) blocks from the free list;
 * pair k of session s is (remote_blk[rem_off[s] + L_loc + k], free_blocks[dst_start[s] + k]).
 * Returns 0, 5 if the free list is too short (decisions written, no pairs), or -1 on allocation
 * failure.
 */
#define ORACLE_MATCH_FILL_HOLES 1
#define ORACLE_MATCH_KEEP_LAST 2

int oracle_match_ex(int32_t n_sessions, const uint32_t *tokens, const int64_t *tok_off, int32_t block_size,
                    const uint64_t *local_keys, int64_t n_local, const uint64_t *remote_hash,
                    const int32_t *remote_blk, const int64_t *rem_off, int32_t threshold,
                    const int32_t *free_blocks, int64_t n_free, int32_t flags, const int64_t *expiry, int64_t now,
                    int32_t *out_local_hit, int32_t *out_remote_hit, int32_t *out_missing, int32_t *out_push,
                    int64_t *out_dst_start, int32_t *pair_src, int32_t *pair_dst, int64_t *n_pairs)
{
    uint64_t *sorted = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_local > 0 ? n_local : 1));
    if (!sorted) return -1;
    memcpy(sorted, local_keys, sizeof(uint64_t) * (size_t)n_local);
    qsort(sorted, (size_t)n_local, sizeof(uint64_t), oracle_cmp_u64);

    for (int32_t s = 0; s < n_sessions; ++s) {
        int64_t n_tok = tok_off[s + 1] - tok_off[s];
        int64_t n_full = n_tok / block_size;
        uint64_t *h = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_full > 0 ? n_full : 1));
        if (!h) { free(sorted); return -1; }
        oracle_block_hashes(tokens + tok_off[s], n_tok, block_size, h);

        int64_t l_loc = 0;
        while (l_loc < n_full && oracle_is_resident(sorted, n_local, h[l_loc])) ++l_loc;

        int64_t n_rem = rem_off[s + 1] - rem_off[s];
        if (expiry && now >= expiry[s]) n_rem = 0;                 /* retention expired */
        int64_t l_rem = 0;
        while (l_rem < n_full && l_rem < n_rem && h[l_rem] == remote_hash[rem_off[s] + l_rem]) ++l_rem;
        if ((flags & ORACLE_MATCH_KEEP_LAST) && l_rem > 0 && l_rem * block_size >= n_tok) --l_rem;

        int64_t missing_blocks = l_rem > l_loc ? l_rem - l_loc : 0;
        if (flags & ORACLE_MATCH_FILL_HOLES) {
            missing_blocks = 0;
            for (int64_t j = 0; j < l_rem; ++j)
                if (!oracle_is_resident(sorted, n_local, h[j])) ++missing_blocks;
        }
        free(h);
        int64_t missing = missing_blocks * block_size;
        out_local_hit[s] = (int32_t)l_loc;
        out_remote_hit[s] = (int32_t)l_rem;
        out_missing[s] = (int32_t)missing;
        out_push[s] = (missing > 0 && missing >= threshold) ? 1 : 0;
    }

    int64_t cursor = 0;
    for (int32_t s = 0; s < n_sessions; ++s) {
        if (out_push[s]) {
            out_dst_start[s] = cursor;
            cursor += out_missing[s] / block_size;
        } else {
            out_dst_start[s] = -1;
        }
    }
    if (cursor > n_free) {
        free(sorted);
        *n_pairs = 0;
        return 5;
    }
    int64_t k = 0;
    for (int32_t s = 0; s < n_sessions; ++s) {
        if (!out_push[s]) continue;
        if (flags & ORACLE_MATCH_FILL_HOLES) {
            /* the non-resident blocks of [0, L_rem), in order */
            int64_t n_tok = tok_off[s + 1] - tok_off[s];
            int64_t n_full = n_tok / block_size;
            uint64_t *h = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_full > 0 ? n_full : 1));
            if (!h) { free(sorted); return -1; }
            oracle_block_hashes(tokens + tok_off[s], n_tok, block_size, h);
            int64_t i = 0;
            for (int64_t j = 0; j < out_remote_hit[s]; ++j) {
                if (oracle_is_resident(sorted, n_local, h[j])) continue;
                pair_src[k] = remote_blk[rem_off[s] + j];
                pair_dst[k] = free_blocks[out_dst_start[s] + i];
                ++k;
                ++i;
            }
            free(h);
            continue;
        }
        int64_t nb = out_missing[s] / block_size;
        for (int64_t i = 0; i < nb; ++i) {
            pair_src[k] = remote_blk[rem_off[s] + out_local_hit[s] + i];
            pair_dst[k] = free_blocks[out_dst_start[s] + i];
            ++k;
        }
    }
    free(sorted);
    *n_pairs = k;
    return 0;
}

int oracle_match(int32_t n_sessions, const uint32_t *tokens, const int64_t *tok_off, int32_t block_size,
                 const uint64_t *local_keys, int64_t n_local, const uint64_t *remote_hash,
                 const int32_t *remote_blk, const int64_t *rem_off, int32_t threshold,
                 const int32_t *free_blocks, int64_t n_free, int32_t *out_local_hit,
                 int32_t *out_remote_hit, int32_t *out_missing, int32_t *out_push, int64_t *out_dst_start,
                 int32_t *pair_src, int32_t *pair_dst, int64_t *n_pairs)
{
    return oracle_match_ex(n_sessions, tokens, tok_off, block_size, local_keys, n_local, remote_hash, remote_blk,
                           rem_off, threshold, free_blocks, n_free, 0, NULL, 0, out_local_hit, out_remote_hit,
                           out_missing, out_push, out_dst_start, pair_src, pair_dst, n_pairs);
}
