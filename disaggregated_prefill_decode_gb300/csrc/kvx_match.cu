// Bidirectional reuse on the device: chained block hashes, the resident-block hash table, the
// per-session match with the recompute threshold, and emission of the decode->prefill copy plan.
//
// Follows the bidirectional KV transfer article (spke.com 3845): Figure 1 steps 4-6 (prefill checks
// the remote reusable KV after applying local cache hits, queues a receive when the reusable tokens
// reach the threshold, then the transfer moves decode blocks to prefill) and "KV-Recompute-
// Schwellenwert" (recompute below the threshold, pull at or above it). The block hash is chained
// 64-bit FNV-1a (Fowler/Noll/Vo): per octet, xor then multiply by the FNV prime.
#include "kvx_internal.h"

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <new>

namespace kvx {

constexpr uint64_t kFnvBasis = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;
static_assert(kFnvPrime == (1ull << 40) + 0x1b3u, "fnv_step splits the prime as 2^40 + 0x1b3");

// ------------------------------------------------------------------------------------------------
// Hashing
// ------------------------------------------------------------------------------------------------

// One FNV-1a step on the hash held as two 32-bit halves. The prime is 2^40 + 0x1b3, so with
// t = lo ^ b: (hi:lo ^ b) * prime mod 2^64 = hi':lo' where lo' = t * 0x1b3 mod 2^32 and
// hi' = hi * 0x1b3 + high word of (t * 0x1b3) + (t << 8) mod 2^32. The low half is the only chain
// that depends on itself alone (xor, 32-bit multiply); the high half follows it.
__device__ __forceinline__ void fnv_step(uint32_t &lo, uint32_t &hi, uint32_t byte) {
    const uint32_t t = lo ^ byte;
    lo = t * 0x1b3u;
    hi = hi * 0x1b3u + __umulhi(t, 0x1b3u) + (t << 8);
}

__device__ __forceinline__ void fnv_word(uint32_t &lo, uint32_t &hi, uint32_t v) {
    fnv_step(lo, hi, v & 0xffu);
    fnv_step(lo, hi, (v >> 8) & 0xffu);
    fnv_step(lo, hi, (v >> 16) & 0xffu);
    fnv_step(lo, hi, v >> 24);
}

constexpr uint32_t kFnvBasisLo = (uint32_t)kFnvBasis, kFnvBasisHi = (uint32_t)(kFnvBasis >> 32);
constexpr unsigned kFull = 0xffffffffu;

// Walks one session's full blocks with a whole warp. The session's tokens are a flat stream of
// n_full * bs ids; the warp loads 64 of them at a time (two per lane, coalesced), loading the next 64
// while the current ones are hashed, and every lane runs the same chain, taking each token from its
// owner lane by shuffle. After each block every lane holds its hash h and calls on_block(j, h).
// on_block returns false to stop early. All branches are uniform across the warp.
// `parent` is the hash the first block chains to (0 for a session's first block).
template <typename OnBlock>
__device__ __forceinline__ void warp_chain(const uint32_t *tok, int64_t n_full, int32_t bs, OnBlock &&on_block,
                                           uint64_t parent = 0) {
    const int lane = threadIdx.x & 31;
    const int64_t total = n_full * bs;
    uint32_t nxt_a = 0, nxt_b = 0;
    if (2 * lane < total) nxt_a = tok[2 * lane];
    if (2 * lane + 1 < total) nxt_b = tok[2 * lane + 1];
    uint32_t lo = kFnvBasisLo, hi = kFnvBasisHi;
    int64_t j = 0;
    if ((bs & 63) == 0) {
        // block sizes that are multiples of 64: each chunk of 64 tokens lies inside one block, so the
        // 256 byte steps of a chunk run without a branch
        const int64_t per_block = bs >> 6;
        int64_t chunk_in_block = 0;
        for (int64_t base = 0; base < total; base += 64) {
            const uint32_t a = nxt_a, b = nxt_b;
            const int64_t nb = base + 64;
            if (nb + 2 * lane < total) nxt_a = tok[nb + 2 * lane];
            if (nb + 2 * lane + 1 < total) nxt_b = tok[nb + 2 * lane + 1];
            if (chunk_in_block == 0) {
                lo = kFnvBasisLo;
                hi = kFnvBasisHi;
                fnv_word(lo, hi, (uint32_t)parent);
                fnv_word(lo, hi, (uint32_t)(parent >> 32));
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) fnv_word(lo, hi, __shfl_sync(kFull, (i & 1) ? b : a, i >> 1));
            if (++chunk_in_block == per_block) {
                chunk_in_block = 0;
                parent = ((uint64_t)hi << 32) | lo;
                if (!on_block(j, parent)) return;
                ++j;
            }
        }
        return;
    }
    int32_t in_block = 0;
    for (int64_t base = 0; base < total; base += 64) {
        const uint32_t a = nxt_a, b = nxt_b;
        const int64_t nb = base + 64;
        if (nb + 2 * lane < total) nxt_a = tok[nb + 2 * lane];
        if (nb + 2 * lane + 1 < total) nxt_b = tok[nb + 2 * lane + 1];
        const int n_here = (int)min((int64_t)64, total - base);
#pragma unroll 8
        for (int i = 0; i < n_here; ++i) {
            const uint32_t v = __shfl_sync(kFull, (i & 1) ? b : a, i >> 1);
            if (in_block == 0) {
                lo = kFnvBasisLo;
                hi = kFnvBasisHi;
                fnv_word(lo, hi, (uint32_t)parent);
                fnv_word(lo, hi, (uint32_t)(parent >> 32));
            }
            fnv_word(lo, hi, v);
            if (++in_block == bs) {
                in_block = 0;
                parent = ((uint64_t)hi << 32) | lo;
                if (!on_block(j, parent)) return;
                ++j;
            }
        }
    }
}

// One warp per session; hashes go out a window of 32 blocks at a time (lane k writes block k of the
// window), coalesced. The first block chains to parent[s] (0 without a parent array).
__global__ void __launch_bounds__(128) kvx_hash_sessions(const uint32_t *tokens, const int64_t *tok_off,
                                                         int32_t n_sessions, int32_t bs, const uint64_t *parent,
                                                         uint64_t *out, const int64_t *hash_off,
                                                         int32_t *err) {
    const int32_t s = (int32_t)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= n_sessions) return;
    const int64_t n_tok_total = tok_off[n_sessions];             // the CSR's own total bounds every read
    const int64_t t0 = tok_off[s], n_tok = tok_off[s + 1] - t0;
    const int64_t n_full = n_tok > 0 ? n_tok / bs : 0;
    if (t0 < 0 || n_tok < 0 || t0 + n_tok > n_tok_total || hash_off[s] < 0 || hash_off[s + 1] - hash_off[s] < n_full) {
        if (lane == 0) atomicOr(err, 1);
        return;
    }
    uint64_t *o = out + hash_off[s];
    uint64_t mine = 0;
    warp_chain(tokens + t0, n_full, bs, [&](int64_t j, uint64_t h) {
        if ((j & 31) == lane) mine = h;
        if ((j & 31) == 31 || j == n_full - 1) {
            const int64_t w0 = j & ~(int64_t)31;
            if (w0 + lane <= j) o[w0 + lane] = mine;
        }
        return true;
    }, parent ? parent[s] : 0);
}

// ------------------------------------------------------------------------------------------------
// Resident-block table: open addressing, linear probing, key 0 kept in the header
// ------------------------------------------------------------------------------------------------

struct TableHeader {
    int32_t has_zero;
    int32_t zero_val;
    int32_t dup;
    int32_t pad;
};

struct TableView {
    const uint64_t *keys;
    const int32_t *vals;
    const TableHeader *hdr;
    uint64_t mask;
    int32_t shift;
};

__device__ __forceinline__ uint64_t slot_of(uint64_t key, int32_t shift) {
    return (key * 0x9E3779B97F4A7C15ull) >> shift;
}

__global__ void kvx_table_insert(const uint64_t *keys, const int32_t *vals, int64_t n, uint64_t *tkeys, int32_t *tvals,
                                 TableHeader *hdr, uint64_t mask, int32_t shift) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint64_t k = keys[i];
    const int32_t v = vals[i];
    if (k == 0) {
        if (atomicExch(&hdr->has_zero, 1) == 1) atomicExch(&hdr->dup, 1);
        hdr->zero_val = v;
        return;
    }
    uint64_t idx = slot_of(k, shift);
    for (uint64_t probe = 0; probe <= mask; ++probe) {
        const unsigned long long prev =
            atomicCAS(reinterpret_cast<unsigned long long *>(tkeys + idx), 0ull, (unsigned long long)k);
        if (prev == 0ull) { tvals[idx] = v; return; }
        if (prev == (unsigned long long)k) { atomicExch(&hdr->dup, 1); return; }
        idx = (idx + 1) & mask;
    }
    atomicExch(&hdr->dup, 2);   // table full: cannot happen at load factor <= 1/2
}

__device__ __forceinline__ int32_t table_find(const TableView &t, uint64_t key) {
    if (key == 0) return t.hdr->has_zero ? t.hdr->zero_val : -1;
    uint64_t idx = slot_of(key, t.shift);
    for (uint64_t probe = 0; probe <= t.mask; ++probe) {
        const uint64_t k = t.keys[idx];
        if (k == key) return t.vals[idx];
        if (k == 0) return -1;
        idx = (idx + 1) & t.mask;
    }
    return -1;
}

__global__ void kvx_table_lookup_kernel(TableView t, const uint64_t *keys, int64_t n, int32_t *out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = table_find(t, keys[i]);
}

// ------------------------------------------------------------------------------------------------
// Match
// ------------------------------------------------------------------------------------------------

// Options of the match on the device (kvx_match_opts plus the hole-filling scratch).
struct MatchFlags {
    int32_t flags;           // KVX_MATCH_*
    const int64_t *expiry;   // per session, or NULL
    int64_t now;
    uint8_t *resident;       // FILL_HOLES: per published block, 1 if resident locally (scratch)
};

// Hash of one block chained to `parent`: the 8 parent octets, then the block's token octets. The
// tokens are read 16 bytes at a time where aligned: a scalar head up to the first 16-byte boundary,
// the aligned body, a scalar tail.
__device__ __forceinline__ uint64_t block_hash(uint64_t parent, const uint32_t *tok, int32_t bs) {
    uint32_t lo = kFnvBasisLo, hi = kFnvBasisHi;
    fnv_word(lo, hi, (uint32_t)parent);
    fnv_word(lo, hi, (uint32_t)(parent >> 32));
    const int32_t head = min(bs, (int32_t)((16 - ((uintptr_t)tok & 15)) & 15) >> 2);
    for (int32_t i = 0; i < head; ++i) fnv_word(lo, hi, __ldg(tok + i));
    const uint4 *v = reinterpret_cast<const uint4 *>(tok + head);
    const int32_t n_vec = (bs - head) >> 2;
#pragma unroll 4
    for (int32_t i = 0; i < n_vec; ++i) {
        const uint4 q = __ldg(v + i);
        fnv_word(lo, hi, q.x);
        fnv_word(lo, hi, q.y);
        fnv_word(lo, hi, q.z);
        fnv_word(lo, hi, q.w);
    }
    for (int32_t i = head + 4 * n_vec; i < bs; ++i) fnv_word(lo, hi, __ldg(tok + i));
    return ((uint64_t)hi << 32) | lo;
}

// ------------------------------------------------------------------------------------------------
// Scans: warp shuffles inside a warp, warp totals through shared memory; across blocks a single
// pass that looks back over the earlier tiles (kvx_scan_lookback, below).
// ------------------------------------------------------------------------------------------------

constexpr int kScanThreads = 1024;

// Inclusive scan of one value per thread across the block; returns it and the block total.
__device__ __forceinline__ int64_t block_inclusive_scan(int64_t v, int64_t *warp_sums, int64_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < n_warps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    *total = warp_sums[n_warps - 1];
    __syncthreads();
    return v;
}

// 512 threads: two CTAs per SM at 62 registers, so 304 sessions are resident at once; measured on
// GB300 against 256 threads (one round of candidates fewer for sessions past 256 blocks: 0.054 ms
// against 0.061 ms per 256-session call) and against two candidates per thread (0.063-0.064 ms: the
// second chain doubles the work of the many sessions shorter than a round).
constexpr int kMatchThreads = 512;

// One CTA per session. The remote prefix is found without walking the chain: block j is hashed from
// the PUBLISHED hash of block j - 1 (its candidate c_j), and the first j where c_j differs from the
// published hash is exactly the first j where the session's own chained hash h_j does: below it every
// published parent equals the true one, so c_j = h_j, and at it the parent is still the true one,
// so c_j = h_j there too. The candidates are independent, so the CTA hashes 512 of them at a time
// (one per thread), each also looked up in the table; each warp then summarises its window of 32
// with ballots and warp 0 extends the two prefixes over the windows in one pass. Local hits can use candidates up to and including the first mismatch; if every
// block to there is resident, warp 0 continues the true chain from that block, window by window, until
// the first block that is not resident. With FILL_HOLES, residency inside the remote prefix is
// recorded for the plan emission and the non-resident blocks there are counted.
__global__ void __launch_bounds__(kMatchThreads, 2) kvx_match_sessions(const uint32_t *tokens, const int64_t *tok_off,
                                                                    int32_t n_sessions, int32_t bs, TableView table,
                                                                    const uint64_t *remote_hash, const int64_t *rem_off,
                                                                    int32_t threshold, MatchFlags mf, kvx_match_result *out,
                                                                    int64_t *push_blocks, int64_t *sess_start,
                                                                    int64_t *scalars, int64_t n_free, int32_t *err) {
    __shared__ uint64_t cand[kMatchThreads];
    __shared__ uint8_t flag[kMatchThreads];     // bit 0: equals the published hash, bit 1: resident
    __shared__ int32_t win_fr[kMatchThreads / 32], win_fl[kMatchThreads / 32], win_holes[kMatchThreads / 32];
    __shared__ int32_t go_on, is_last;
    __shared__ int64_t scan_ws[32];
    const int32_t s = (int32_t)blockIdx.x;
    if (s >= n_sessions) return;                                  // never: the grid is one CTA per session
    const int tid = (int)threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the two CSR totals bound every read of the token and published-hash arrays
    const int64_t n_tok_total = tok_off[n_sessions], n_pub = rem_off[n_sessions];
    int64_t t0 = tok_off[s], n_tok = tok_off[s + 1] - t0;
    int64_t r0 = rem_off[s], n_rem = rem_off[s + 1] - r0;
    // malformed offsets: flag them and treat the session as empty, so no array is read out of range
    if (t0 < 0 || n_tok < 0 || t0 + n_tok > n_tok_total) {
        if (tid == 0) atomicOr(err, 1);
        t0 = 0;
        n_tok = 0;
    }
    if (r0 < 0 || n_rem < 0 || r0 + n_rem > n_pub) {
        if (tid == 0) atomicOr(err, 2);
        r0 = 0;
        n_rem = 0;
    }
    if (mf.expiry && mf.now >= mf.expiry[s]) n_rem = 0;           // retention expired
    const bool fill = (mf.flags & KVX_MATCH_FILL_HOLES) != 0;
    const int64_t n_full = n_tok > 0 ? n_tok / bs : 0;
    const int64_t n_cand = min(n_full, n_rem + 1);                // the published blocks and the one after
    const uint32_t *tk = tokens + t0;
    // warp 0's state (uniform across its lanes)
    int64_t l_loc = 0, l_rem = 0, holes = 0;
    bool loc_open = true, rem_open = true, chain = false;
    uint64_t chain_parent = 0;
    for (int64_t base = 0; base < n_cand; base += kMatchThreads) {
        const int64_t j = base + tid;
        if (j < n_cand) {
            const uint64_t c = block_hash(j == 0 ? 0 : remote_hash[r0 + j - 1], tk + j * bs, bs);
            const bool same = j < n_rem && remote_hash[r0 + j] == c;
            const bool res = table_find(table, c) >= 0;
            cand[tid] = c;
            flag[tid] = (uint8_t)((same ? 1 : 0) | (res ? 2 : 0));
        }
        __syncthreads();
        // every warp summarises its window of 32 candidates: the first published-hash mismatch, the
        // first block not resident, and (hole filling) the non-resident blocks before the mismatch
        {
            const int64_t j0 = base + 32 * warp;
            const uint8_t f = j0 + lane < n_cand ? flag[tid] : 0;     // past the candidates: both miss
            const unsigned hit = __ballot_sync(kFull, f & 2);
            const unsigned rmiss = ~__ballot_sync(kFull, f & 1);
            const int fr = rmiss ? __ffs(rmiss) - 1 : 32;
            const int fl = ~hit ? __ffs(~hit) - 1 : 32;
            // residency below the window's first mismatch. Every round that runs starts with the remote
            // prefix open (once it closes, the local one has closed too); entries past the remote
            // prefix are written as well and never read (the emission looks only below it)
            if (fill && lane < fr) mf.resident[r0 + j0 + lane] = (f & 2) ? 1 : 0;
            if (lane == 0) {
                win_fr[warp] = fr;
                win_fl[warp] = fl;
                win_holes[warp] = __popc(~hit & (fr >= 32 ? kFull : ((1u << fr) - 1u)));
            }
        }
        __syncthreads();
        if (warp == 0) {
            // the windows in order, one lane each: the remote prefix runs to the first window with a
            // mismatch; local hits run while resident, up to and including the first mismatch block
            // (whose candidate is still its true hash)
            constexpr int kWin = kMatchThreads / 32;
            const bool valid = lane < kWin;
            const int fr = valid ? win_fr[lane] : 32, fl = valid ? win_fl[lane] : 32;
            const int hw = valid ? win_holes[lane] : 0;
            int wr = kWin, fr_w = 32;                                   // first window with a mismatch
            const bool rem_was_open = rem_open;
            if (rem_open) {
                const unsigned m = __ballot_sync(kFull, valid && fr < 32);
                wr = m ? __ffs(m) - 1 : kWin;
                fr_w = __shfl_sync(kFull, fr, wr < kWin ? wr : 0);
                if (fill) {
                    int h = lane <= wr ? hw : 0;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(kFull, h, o);
                    holes += h;
                }
                l_rem += 32 * wr + (wr < kWin ? fr_w : 0);
                rem_open = wr == kWin;
            }
            if (loc_open) {
                // positions of window w local hits may use: all before wr, through the mismatch at wr
                const int lim = !rem_was_open ? 0 : lane < wr ? 32 : (lane == wr ? fr_w + 1 : 0);
                const unsigned m = __ballot_sync(kFull, valid && fl < lim);
                const int wl = m ? __ffs(m) - 1 : kWin;
                if (wl < kWin && wl <= wr) {
                    l_loc += 32 * wl + __shfl_sync(kFull, fl, wl);
                    loc_open = false;
                } else if (!rem_was_open) {
                    loc_open = false;
                } else if (wr < kWin) {                                 // resident through the mismatch
                    l_loc += 32 * wr + fr_w + 1;
                    loc_open = false;
                    chain = true;
                    chain_parent = cand[32 * wr + fr_w];
                } else {
                    l_loc += 32 * kWin;
                }
            }
            if (lane == 0) go_on = rem_open || loc_open;
        }
        __syncthreads();
        if (!go_on) break;
    }
    if (warp == 0 && chain && l_loc < n_full) {
        // beyond the first mismatch the published parents no longer hold: the true chain, from the
        // candidate of that block, while the blocks stay resident (looked up 32 at a time)
        uint64_t mine = 0;
        const int64_t jb = l_loc;
        bool open = true;
        warp_chain(tk + jb * bs, n_full - jb, bs, [&](int64_t k, uint64_t h) {
            if ((k & 31) == lane) mine = h;
            if ((k & 31) != 31 && k != n_full - jb - 1) return true;
            const int n_valid = (int)(k - (k & ~(int64_t)31) + 1);
            const bool hit = lane < n_valid && table_find(table, mine) >= 0;
            const unsigned miss = ~__ballot_sync(kFull, hit);
            const int fl = miss ? __ffs(miss) - 1 : 32;
            l_loc += min(fl, n_valid);
            open = fl >= n_valid;
            return open;
        }, chain_parent);
    }
    if (tid == 0) {                                               // the session's result
        if ((mf.flags & KVX_MATCH_KEEP_LAST) && l_rem > 0 && l_rem * bs >= n_tok) {
            // every token is covered (the session ends on a block boundary and its whole chain matched):
            // recompute the last block
            --l_rem;
            if (fill && !mf.resident[r0 + l_rem]) --holes;
        }
        const int64_t missing_blocks = fill ? holes : (l_rem > l_loc ? l_rem - l_loc : 0);
        const int64_t missing = missing_blocks * bs;
        if (missing > (int64_t)INT32_MAX || l_loc > (int64_t)INT32_MAX) atomicOr(err, 4);
        const int32_t push = (missing > 0 && missing >= threshold) ? 1 : 0;
        kvx_match_result r;
        r.local_hit_blocks = (int32_t)l_loc;
        r.remote_hit_blocks = (int32_t)l_rem;
        r.missing_tokens = (int32_t)missing;
        r.push = push;
        r.dst_start = -1;
        out[s] = r;
        push_blocks[s] = push ? missing_blocks : 0;
        __threadfence();                                              // visible before this CTA is counted
        is_last = atomicAdd(reinterpret_cast<unsigned long long *>(&scalars[7]), 1ull) ==
                  (unsigned long long)(n_sessions - 1);
    }
    __syncthreads();
    if (!is_last) return;
    // The last CTA to finish: every session's pull count is in. It numbers the pulled blocks in
    // session order (exclusive scan) and hands each pushing session its first free-list position.
    __threadfence();
    int64_t carry = 0;
    for (int32_t b0 = 0; b0 < n_sessions; b0 += kMatchThreads) {
        const int32_t i = b0 + tid;
        const int64_t v = i < n_sessions ? push_blocks[i] : 0;
        int64_t tot;
        const int64_t inc = block_inclusive_scan(v, scan_ws, &tot);
        if (i < n_sessions) sess_start[i] = carry + inc - v;
        carry += tot;
    }
    for (int32_t i = tid; i < n_sessions; i += kMatchThreads)
        if (out[i].push) out[i].dst_start = sess_start[i];
    if (tid == 0) {
        // the pulled blocks never exceed the published ones (else the remote offsets overlap)
        const bool fits = carry <= n_free, sane = carry <= max(n_pub, (int64_t)1);
        scalars[0] = carry;
        scalars[4] = (fits && sane) ? carry : 0;
        if (!sane) atomicOr(err, 2);
        else if (!fits) atomicOr(err, 8);
    }
}

// The whole scan in one block, for n <= kScanThreads.
__global__ void __launch_bounds__(kScanThreads) kvx_scan_single(const int64_t *in, int64_t *out, int64_t n_host,
                                                                 const int64_t *n_dev, int64_t *sum) {
    __shared__ int64_t ws[32];
    const int64_t n = n_dev ? min(*n_dev, n_host) : n_host;   // a device count never past the host bound
    const int64_t i = threadIdx.x;
    const int64_t v = i < n ? in[i] : 0;
    int64_t total;
    const int64_t inc = block_inclusive_scan(v, ws, &total);
    if (i < n) out[i] = inc - v;
    if (threadIdx.x == 0) *sum = total;
}

// Error bit 64: a look-back scan gave up waiting on an earlier tile, so the sums after it are wrong.
// The kernels that consume scan results then do nothing (the call returns KVX_ETIMEDOUT): indexes
// taken from wrong sums could point outside the arrays.
constexpr int32_t kScanTimedOut = 64;
__device__ __forceinline__ bool scan_failed(const int32_t *err) {
    return (*(const volatile int32_t *)err & kScanTimedOut) != 0;
}

constexpr uint64_t kScanWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait on a predecessor
constexpr uint64_t kScanStallWaitNs = 1000000ull;  // 1 ms: the bound under the testing hook

__device__ __forceinline__ uint64_t scan_clock_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Longer scans in one pass, with a look back over the tiles before: a CTA takes the next tile in
// order by an atomic ticket (so every earlier tile belongs to a CTA already running, which never
// waits on a later one), publishes its tile's total, then walks back over the earlier tiles adding
// their totals until it meets one that has published its running prefix, and publishes its own.
// state[t] holds 0 (nothing yet), total * 4 + 1 (the tile's total) or prefix * 4 + 2 (the prefix
// through the tile); state[n_tiles] is the ticket counter; all zero before the launch. A wait is
// bounded by the global timer (wait_ns): past the bound the scan sets error bit 64 and goes on (wrong
// sums, which the kernels after it then leave unused; the caller returns KVX_ETIMEDOUT). stall_tile (testing hook, -1 normally): that tile publishes nothing,
// so the tile after it waits until the bound.
__global__ void __launch_bounds__(kScanThreads) kvx_scan_lookback(const int64_t *in, int64_t *out, int64_t n_host,
                                                                   const int64_t *n_dev, unsigned long long *state,
                                                                   int64_t n_tiles, int64_t *sum, int32_t *err,
                                                                   int64_t stall_tile, uint64_t wait_ns) {
    __shared__ int64_t ws[32];
    __shared__ int64_t tile_s, excl_s;
    if (threadIdx.x == 0) tile_s = (int64_t)atomicAdd(&state[n_tiles], 1ull);
    __syncthreads();
    const int64_t tile = tile_s;
    const int64_t n = n_dev ? min(*n_dev, n_host) : n_host;   // a device count never past the host bound
    const int64_t i = tile * blockDim.x + threadIdx.x;
    const int64_t v = i < n ? in[i] : 0;
    int64_t total;
    const int64_t inc = block_inclusive_scan(v, ws, &total);
    if (threadIdx.x == 0) {
        int64_t excl = 0;
        const bool publish = tile != stall_tile;
        if (tile > 0) {
            if (publish) atomicExch(&state[tile], ((unsigned long long)total << 2) | 1ull);
            uint64_t t0 = 0;
            for (int64_t p = tile - 1;;) {
                const unsigned long long f = __ldcg(&state[p]);             // from L2, where the writers publish
                if ((f & 3ull) == 0) {
                    if (t0 == 0) t0 = scan_clock_ns();
                    else if (scan_clock_ns() - t0 > wait_ns) { atomicOr(err, kScanTimedOut); break; }
                    continue;
                }
                excl += (int64_t)(f >> 2);
                if (f & 2ull) break;
                --p;                                                    // tile 0 always publishes a prefix
                t0 = 0;
            }
        }
        if (publish) atomicExch(&state[tile], ((unsigned long long)(excl + total) << 2) | 2ull);
        excl_s = excl;
        if (tile == n_tiles - 1) *sum = excl + total;
    }
    __syncthreads();
    if (i < n) out[i] = excl_s + inc - v;
}

// Exclusive scan of in[0..n) into out, total into *sum. n_bound is a host upper bound on n; `state`
// holds scan_state_words(n_bound) zeroed words (unused for n_bound <= kScanThreads).
static int64_t scan_state_words(int64_t n_bound) {
    return (n_bound + kScanThreads - 1) / kScanThreads + 1;
}

// stall (testing hook): the look-back scan's first tile publishes nothing and the waits are bounded
// by 1 ms, so the second tile's wait runs out (no effect on a single-tile scan).
static cudaError_t exclusive_scan(const int64_t *in, int64_t *out, int64_t n_bound, const int64_t *n_dev,
                                  unsigned long long *state, int64_t *sum, int32_t *err, cudaStream_t st,
                                  bool stall = false) {
    count_launch(1);
    if (n_bound <= kScanThreads) {
        kvx_scan_single<<<1, kScanThreads, 0, st>>>(in, out, n_bound, n_dev, sum);
        return cudaGetLastError();
    }
    const int64_t nb = scan_state_words(n_bound) - 1;
    kvx_scan_lookback<<<(unsigned)nb, kScanThreads, 0, st>>>(in, out, n_bound, n_dev, state, nb, sum, err,
                                                              stall ? 0 : -1, stall ? kScanStallWaitNs : kScanWaitNs);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Decode -> prefill plan emission
// ------------------------------------------------------------------------------------------------

// Scalars: [0] blocks the pushes need, [1] runs, [2] tiles, [4] blocks the plan emits ([0], or 0
// when the free list is too short), [5] hole-filling pull flags counted, [7] match CTAs finished.
struct MatchScratch {
    int64_t *push_blocks;   // [n_sessions]
    int64_t *sess_start;    // [n_sessions] exclusive scan of push_blocks
    int64_t *pair_src;      // [B] decode block of pushed block k
    int64_t *pair_dst;      // [B] prefill block of pushed block k
    int64_t *flag;          // [B] 1 where a run starts
    int64_t *run_idx;       // [B] exclusive scan of flag
    int64_t *run_start;     // [B] first pushed block of each run
    int64_t *tile_count;    // [B] tiles of each run
    int64_t *tile_start;    // [B] exclusive scan of tile_count
    unsigned long long *scan_state;   // three regions of scan_state_words(B) words: the look-back scans
    int64_t *scalars;       // [8]
    int32_t *err;           // [4] error bits
};


// One thread per pushed block k: its session, its (decode, prefill) pair, and whether it starts a
// run (first block of a session, or either id not its predecessor's + 1).
__global__ void kvx_emit_pairs(const kvx_match_result *res, const int64_t *sess_start, int32_t n_sessions,
                               const int32_t *remote_blk, const int64_t *rem_off, const int32_t *free_blocks,
                               const int64_t *total, int64_t *pair_src, int64_t *pair_dst, int64_t *flag) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= *total) return;
    // The last session whose range starts at or before k owns k: a pushing session s covers
    // [sess_start[s], sess_start[s] + n_s) and every later session starts at or after its end.
    int32_t lo = 0, hi = n_sessions - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (sess_start[mid] <= k) lo = mid; else hi = mid - 1;
    }
    const int32_t s = lo;
    const int64_t i = k - sess_start[s];
    const int64_t base = rem_off[s] + res[s].local_hit_blocks;
    const int64_t src = remote_blk[base + i];
    const int64_t dst = free_blocks[k];
    pair_src[k] = src;
    pair_dst[k] = dst;
    int64_t starts = 1;
    if (i > 0) starts = (src == (int64_t)remote_blk[base + i - 1] + 1 && dst == (int64_t)free_blocks[k - 1] + 1) ? 0 : 1;
    flag[k] = starts;
}

// FILL_HOLES emission, step 1: published block k is pulled when its session pushes, it lies below
// the session's remote prefix and it is not resident locally. Its session comes from a binary search
// over the remote offsets, checked against the session's range (offsets of sessions flagged as
// malformed never push).
__device__ __forceinline__ int32_t session_of(const int64_t *rem_off, int32_t n_sessions, int64_t k) {
    int32_t lo = 0, hi = n_sessions - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (rem_off[mid] <= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void kvx_need_flags(const kvx_match_result *res, const int64_t *rem_off, int32_t n_sessions, int64_t n_pub,
                               const uint8_t *resident, int64_t *need) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_pub) return;
    const int32_t s = session_of(rem_off, n_sessions, k);
    const int64_t j = k - rem_off[s];
    const bool mine = j >= 0 && k < rem_off[s + 1];
    need[k] = (mine && res[s].push && j < res[s].remote_hit_blocks && !resident[k]) ? 1 : 0;
}

// Step 2: pulled block k goes to position npos[k] of the pair list (an exclusive scan of need), the
// free-list entry of the same position; positions past the plan's block count are not emitted.
__global__ void kvx_emit_pairs_holes(const int64_t *need, const int64_t *npos, const int64_t *total,
                                     const int32_t *remote_blk, const int64_t *rem_off, int32_t n_sessions,
                                     int64_t n_pub, const int32_t *free_blocks, int64_t *pair_src, int64_t *pair_dst,
                                     int64_t *pair_sess, const int64_t *n_need, const int64_t *n_counted, int32_t *err) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (scan_failed(err)) return;
    // the flags must account for exactly the blocks the sessions counted
    if (k == 0 && n_pub > 0 && *n_need != *n_counted) atomicOr(err, 32);
    if (k >= n_pub || !need[k]) return;
    const int64_t pos = npos[k];
    if (pos < 0 || pos >= *total) return;
    pair_src[pos] = remote_blk[k];
    pair_dst[pos] = free_blocks[pos];
    pair_sess[pos] = session_of(rem_off, n_sessions, k);
}

// Step 3: a run starts at a new session or where either block id does not continue the previous.
__global__ void kvx_run_flags(const int64_t *pair_src, const int64_t *pair_dst, const int64_t *pair_sess,
                              const int64_t *total, int64_t *flag, const int32_t *err) {
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= *total || scan_failed(err)) return;
    flag[p] = (p == 0 || pair_sess[p] != pair_sess[p - 1] || pair_src[p] != pair_src[p - 1] + 1 ||
               pair_dst[p] != pair_dst[p - 1] + 1) ? 1 : 0;
}

// run_idx[k] is the exclusive scan of the run flags, so a run's number lies in [0, total); one outside
// is reported (bit 16) and not written.
__global__ void kvx_run_starts(const int64_t *flag, const int64_t *run_idx, const int64_t *total, int64_t *run_start,
                               int32_t *err) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= *total || !flag[k] || scan_failed(err)) return;
    const int64_t r = run_idx[k];
    if (r < 0 || r >= *total) { atomicOr(err, 16); return; }
    run_start[r] = k;
}

struct EmitShape {
    int64_t src_row_bytes, dst_row_bytes;
    int32_t bs;
    int32_t strided;
    int32_t tile_bytes;
    int32_t rows_per_tile;
    int32_t n_pairs;
    int32_t per_head;                    // a head-major side: tiles per (block, head)
    int32_t pair_s[8], pair_d[8];
    int64_t pair_soff[8], pair_doff[8];
    // per_head: the head partition and layout of each side, the head's bytes, each side's token and
    // head pitch, heads per tile and the head groups of one block (tiles per block = groups times the
    // row chunks of a head)
    int32_t heads, hps_s, hps_d, layout_s, layout_d, heads_per_tile, groups;
    int64_t head_bytes, src_pitch, dst_pitch, src_head_pitch, dst_head_pitch;
};

// Element index (in heads) of (block, slot 0, head) inside one buffer of a side's layout.
__device__ __forceinline__ int64_t head_start(int32_t layout, int32_t hps, int32_t bs, int64_t blk, int32_t head) {
    return layout == KVX_LAYOUT_HND ? (blk * hps + head) * (int64_t)bs : blk * (int64_t)bs * hps + head;
}

// A run's blocks [run_start[r], run_start[r + 1]) must be a non-empty range inside [0, total): a run
// that is not counts no tiles and is reported (bit 16).
__device__ __forceinline__ bool run_ok(int64_t k0, int64_t k1, int64_t total) { return 0 <= k0 && k0 < k1 && k1 <= total; }

__global__ void kvx_run_tiles(const int64_t *run_start, const int64_t *scalars, EmitShape sh, int64_t *tile_count,
                              int32_t *err) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n_runs = scalars[1], total = scalars[4];
    if (r >= n_runs || scan_failed(err)) return;
    const int64_t k1 = r + 1 < n_runs ? run_start[r + 1] : total;
    if (!run_ok(run_start[r], k1, total)) { tile_count[r] = 0; atomicOr(err, 16); return; }
    const int64_t ntok = (k1 - run_start[r]) * sh.bs;
    if (sh.per_head) {
        tile_count[r] = (k1 - run_start[r]) * sh.groups * ((sh.bs + sh.rows_per_tile - 1) / sh.rows_per_tile);
        return;
    }
    const int64_t per = sh.strided ? (ntok + sh.rows_per_tile - 1) / sh.rows_per_tile
                                   : (ntok * sh.src_row_bytes + sh.tile_bytes - 1) / sh.tile_bytes;
    tile_count[r] = per * sh.n_pairs;
}

// One thread per run: the run's rows (for host introspection) and its tiles, cut as the host plan
// builder cuts them.
__global__ void kvx_emit_tiles(const int64_t *run_start, const int64_t *tile_start, const int64_t *scalars,
                               const int64_t *pair_src, const int64_t *pair_dst, EmitShape sh, TileDesc *tiles,
                               int64_t tile_cap, int32_t *run_src_row, int32_t *run_dst_row, int32_t *run_ntok,
                               int32_t *err) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n_runs = scalars[1], total = scalars[4];
    if (r >= n_runs || scan_failed(err)) return;
    const int64_t k0 = run_start[r];
    const int64_t k1 = r + 1 < n_runs ? run_start[r + 1] : total;
    if (!run_ok(k0, k1, total) || tile_start[r] < 0) { atomicOr(err, 16); return; }
    const int64_t ntok = (k1 - k0) * sh.bs;
    const int64_t srow = pair_src[k0] * sh.bs, drow = pair_dst[k0] * sh.bs;
    run_src_row[r] = (int32_t)srow;
    run_dst_row[r] = (int32_t)drow;
    run_ntok[r] = (int32_t)ntok;
    int64_t t = tile_start[r];
    if (sh.per_head) {
        // every block of the run, by groups of heads that one shard pair shares (as many as fit a
        // tile): bs rows per head at each side's token pitch, the group's heads a head pitch apart
        for (int64_t k = k0; k < k1; ++k)
            for (int32_t g = 0; g < sh.heads;) {
                const int32_t ss = g / sh.hps_s, hs = g % sh.hps_s, ds = g / sh.hps_d, hd = g % sh.hps_d;
                const int32_t kh = min(sh.heads_per_tile, min(sh.hps_s - hs, sh.hps_d - hd));
                const int64_t s0 = head_start(sh.layout_s, sh.hps_s, sh.bs, pair_src[k], hs) * sh.head_bytes;
                const int64_t d0 = head_start(sh.layout_d, sh.hps_d, sh.bs, pair_dst[k], hd) * sh.head_bytes;
                for (int32_t r0 = 0; r0 < sh.bs; r0 += sh.rows_per_tile, ++t) {
                    if (t >= tile_cap) { atomicOr(err, 16); return; }
                    TileDesc d;
                    d.src_off = s0 + r0 * sh.src_pitch;
                    d.dst_off = d0 + r0 * sh.dst_pitch;
                    d.n = min(sh.rows_per_tile, sh.bs - r0);
                    d.s_shard = ss;
                    d.d_shard = ds;
                    d.heads = kh > 1 ? kh : 0;
                    tiles[t] = d;
                }
                g += kh;
            }
        return;
    }
    if (!sh.strided) {
        const int64_t bytes = ntok * sh.src_row_bytes;
        const int64_t s0 = srow * sh.src_row_bytes, d0 = drow * sh.dst_row_bytes;
        for (int64_t o = 0; o < bytes; o += sh.tile_bytes)
            for (int32_t q = 0; q < sh.n_pairs; ++q, ++t) {
                if (t >= tile_cap) { atomicOr(err, 16); return; }
                TileDesc d;
                d.src_off = s0 + o;
                d.dst_off = d0 + o;
                d.n = (int32_t)min((int64_t)sh.tile_bytes, bytes - o);
                d.s_shard = sh.pair_s[q];
                d.d_shard = sh.pair_d[q];
                d.heads = 0;
                tiles[t] = d;
            }
    } else {
        for (int64_t r0 = 0; r0 < ntok; r0 += sh.rows_per_tile)
            for (int32_t q = 0; q < sh.n_pairs; ++q, ++t) {
                if (t >= tile_cap) { atomicOr(err, 16); return; }
                TileDesc d;
                d.src_off = (srow + r0) * sh.src_row_bytes + sh.pair_soff[q];
                d.dst_off = (drow + r0) * sh.dst_row_bytes + sh.pair_doff[q];
                d.n = (int32_t)min((int64_t)sh.rows_per_tile, ntok - r0);
                d.s_shard = sh.pair_s[q];
                d.d_shard = sh.pair_d[q];
                d.heads = 0;
                tiles[t] = d;
            }
    }
}

static unsigned grid_for(int64_t n, int threads) {
    return (unsigned)std::max<int64_t>(1, (n + threads - 1) / threads);
}

}  // namespace kvx

using namespace kvx;

struct kvx_table_s {
    void *dev = nullptr;
    uint64_t *keys = nullptr;
    int32_t *vals = nullptr;
    TableHeader *hdr = nullptr;
    uint64_t capacity = 0;
    int32_t shift = 0;
    int64_t n = 0;
    cudaEvent_t last_use = nullptr;   // recorded after each lookup; destroy waits for it
    int32_t device = -1;              // device of the table, current while it is destroyed
    TableView view() const { return TableView{keys, vals, hdr, capacity - 1, shift}; }
};

extern "C" {

kvx_status kvx_block_hashes(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions, int32_t block_size,
                            uint64_t *out_hash, const int64_t *hash_off, cudaStream_t stream) {
    return kvx_block_hashes_ex(tokens, tok_off, n_sessions, block_size, nullptr, out_hash, hash_off, stream);
}

kvx_status kvx_block_hashes_ex(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions, int32_t block_size,
                               const uint64_t *parent, uint64_t *out_hash, const int64_t *hash_off,
                               cudaStream_t stream) {
    if (n_sessions < 0 || block_size < 1) return fail(KVX_EINVAL, "n_sessions >= 0 and block_size >= 1");
    if (n_sessions == 0) return KVX_OK;
    if (!tokens || !tok_off || !out_hash || !hash_off) return fail(KVX_EINVAL, "NULL device array");
    void *errp = nullptr;
    kvx_status st = pool_alloc(&errp, sizeof(int32_t), stream);
    if (st) return st;
    int32_t *err = static_cast<int32_t *>(errp);
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int32_t), stream);
    if (e == cudaSuccess) {
        count_launch();
        kvx_hash_sessions<<<grid_for((int64_t)n_sessions * 32, 128), 128, 0, stream>>>(tokens, tok_off, n_sessions, block_size,
                                                                       parent, out_hash, hash_off, err);
        e = cudaGetLastError();
    }
    int32_t h_err = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h_err, err, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    pool_free(errp);
    if (e != cudaSuccess) return cuda_fail(e, "kvx_block_hashes");
    if (h_err) return fail(KVX_ERANGE, "malformed tok_off, or a hash_off range shorter than the session's full blocks");
    return KVX_OK;
}

kvx_status kvx_table_build(const uint64_t *keys, const int32_t *vals, int64_t n, cudaStream_t stream, kvx_table_t *out) {
    if (!out) return fail(KVX_EINVAL, "out is NULL");
    *out = nullptr;
    if (n < 0 || (n > 0 && (!keys || !vals))) return fail(KVX_EINVAL, "bad key/value arrays");
    if (n > ((int64_t)1 << 40)) return fail(KVX_EUNSUPPORTED, "table too large");
    kvx_table_s *t = new (std::nothrow) kvx_table_s();
    if (!t) return fail(KVX_ENOMEM, "host allocation failed");
    uint64_t cap = 16;
    int32_t bits = 4;
    while (cap < (uint64_t)(2 * n)) { cap <<= 1; ++bits; }
    t->capacity = cap;
    t->shift = 64 - bits;
    t->n = n;
    const size_t off_vals = align_up(sizeof(uint64_t) * cap, 256);
    const size_t off_hdr = off_vals + align_up(sizeof(int32_t) * cap, 256);
    const size_t bytes = off_hdr + 256;
    if (cudaGetDevice(&t->device) != cudaSuccess) t->device = -1;
    kvx_status st = pool_alloc(&t->dev, bytes, stream);
    if (st) { delete t; return st; }
    t->keys = static_cast<uint64_t *>(t->dev);
    t->vals = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(t->dev) + off_vals);
    t->hdr = reinterpret_cast<TableHeader *>(static_cast<uint8_t *>(t->dev) + off_hdr);
    cudaError_t e = cudaMemsetAsync(t->dev, 0, bytes, stream);
    if (e == cudaSuccess && n > 0) {
        count_launch();
        kvx_table_insert<<<grid_for(n, 256), 256, 0, stream>>>(keys, vals, n, t->keys, t->vals, t->hdr, cap - 1,
                                                               t->shift);
        e = cudaGetLastError();
    }
    TableHeader h = {};
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, t->hdr, sizeof(h), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) { pool_free(t->dev); delete t; return cuda_fail(e, "kvx_table_build"); }
    if (h.dup) { pool_free(t->dev); delete t; return fail(KVX_EINVAL, "duplicate key in table input"); }
    *out = t;
    return KVX_OK;
}

kvx_status kvx_table_lookup(kvx_table_t t, const uint64_t *keys, int64_t n, int32_t *out_vals, cudaStream_t stream) {
    if (!t) return fail(KVX_EINVAL, "NULL table");
    if (n < 0 || (n > 0 && (!keys || !out_vals))) return fail(KVX_EINVAL, "bad arrays");
    if (n == 0) return KVX_OK;
    count_launch();
    kvx_table_lookup_kernel<<<grid_for(n, 256), 256, 0, stream>>>(t->view(), keys, n, out_vals);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && !t->last_use) e = cudaEventCreateWithFlags(&t->last_use, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(t->last_use, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvx_table_lookup");
    return KVX_OK;
}

kvx_status kvx_table_destroy(kvx_table_t t) {
    if (!t) return KVX_OK;
    const DeviceScope on_device(t->device);
    cudaError_t e = cudaSuccess;
    if (t->last_use) {
        e = cudaEventSynchronize(t->last_use);
        cudaEventDestroy(t->last_use);
    }
    if (t->dev) pool_free(t->dev);
    delete t;
    if (e != cudaSuccess) return cuda_fail(e, "kvx_table_destroy");
    return KVX_OK;
}

kvx_status kvx_match_prefix(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions, int32_t block_size,
                            kvx_table_t table, const uint64_t *remote_hash, const int32_t *remote_blk,
                            const int64_t *rem_off, int32_t threshold, const int32_t *free_blocks, int64_t n_free,
                            const kvx_pool *remote_pool, const kvx_pool *local_pool, kvx_match_result *out,
                            kvx_plan_t *out_plan, cudaStream_t stream) {
    return kvx_match_prefix_ex(tokens, tok_off, n_sessions, block_size, table, remote_hash, remote_blk, rem_off,
                               threshold, free_blocks, n_free, remote_pool, local_pool, nullptr, out, out_plan, stream);
}

kvx_status kvx_match_prefix_ex(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions, int32_t block_size,
                               kvx_table_t table, const uint64_t *remote_hash, const int32_t *remote_blk,
                               const int64_t *rem_off, int32_t threshold, const int32_t *free_blocks, int64_t n_free,
                               const kvx_pool *remote_pool, const kvx_pool *local_pool, const kvx_match_opts *opts,
                               kvx_match_result *out, kvx_plan_t *out_plan, cudaStream_t stream) {
    if (out_plan) *out_plan = nullptr;
    if (n_sessions < 0 || block_size < 1 || n_free < 0) return fail(KVX_EINVAL, "bad counts");
    MatchFlags mf = {0, nullptr, 0, nullptr};
    if (opts) {
        if (opts->reserved0 || opts->reserved[0] || opts->reserved[1] || opts->reserved[2] || opts->reserved[3])
            return fail(KVX_EINVAL, "kvx_match_opts.reserved must be 0");
        if (opts->flags & ~(KVX_MATCH_FILL_HOLES | KVX_MATCH_KEEP_LAST | KVX_MATCH_TEST_SCAN_STALL))
            return fail(KVX_EINVAL, "unknown kvx_match_opts.flags bits");
        mf.flags = opts->flags;
        mf.expiry = opts->expiry;
        mf.now = opts->now;
    }
    const bool fill = (mf.flags & KVX_MATCH_FILL_HOLES) != 0;
    if (!table) return fail(KVX_EINVAL, "NULL table");
    if (n_sessions > 0 && (!tokens || !tok_off || !rem_off || !out || !remote_hash || !remote_blk))
        return fail(KVX_EINVAL, "NULL device array");
    if (n_free > 0 && !free_blocks) return fail(KVX_EINVAL, "NULL free list");

    // the plan's geometry is validated before any device work
    kvx_plan_s *pl = nullptr;
    if (out_plan) {
        pl = new (std::nothrow) kvx_plan_s();
        if (!pl) return fail(KVX_ENOMEM, "host allocation failed");
        kvx_status st = init_plan_geometry(remote_pool, local_pool, nullptr, pl);
        if (st) { delete pl; return st; }
        if (pl->src.block_size != block_size || pl->dst.block_size != block_size) {
            delete pl;
            return fail(KVX_EINVAL, "pool block sizes must equal block_size");
        }
        if (pl->per_head) as_whole_block_copy(pl);                   // identical spans when the layouts agree
        if (!pl->per_head && std::max(pl->src.n_shards, pl->dst.n_shards) > 8) {
            delete pl;
            return fail(KVX_EUNSUPPORTED, "device-built plans support at most 8 shard pairs");
        }
        pl->device_built = true;
    }
    if (n_sessions == 0) {
        if (pl) { finish_plan_shape(pl); *out_plan = pl; }
        return KVX_OK;
    }

    // The kernels bound their reads by the CSR totals themselves. Only a plan, or hole filling, needs
    // the published-block count on the host, to size the per-block scratch; a decision-only call
    // does not wait for it.
    int64_t n_pub = 0;
    cudaError_t e = cudaSuccess;
    if (pl || fill) {
        e = cudaMemcpyAsync(&n_pub, rem_off + n_sessions, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) { delete pl; return cuda_fail(e, "reading rem_off"); }
        if (n_pub < 0) { delete pl; return fail(KVX_EINVAL, "rem_off is not a CSR offset array"); }
    }
    const int64_t B = std::max<int64_t>(n_pub, 1);
    const int64_t n_state = scan_state_words(B);

    // scratch, one allocation
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_push = take(sizeof(int64_t) * n_sessions), o_sess = take(sizeof(int64_t) * n_sessions);
    const size_t o_ps = take(8 * B), o_pd = take(8 * B), o_flag = take(8 * B), o_ridx = take(8 * B);
    const size_t o_rstart = take(8 * B), o_tcount = take(8 * B), o_tstart = take(8 * B);
    // scalars [8] and error words [4] side by side: one memset, one read-back
    // scalars [8] and error words [4] side by side, then the scans' look-back state: one memset
    const size_t o_scal = take(8 * 8 + sizeof(int32_t) * 4 + 8 * 3 * n_state), o_err = o_scal + 8 * 8;
    const size_t o_state = o_err + sizeof(int32_t) * 4;
    // hole filling: residency per published block, pull flags, their scan, each pair's session
    const size_t o_res = fill ? take(B) : 0, o_need = fill ? take(8 * B) : 0, o_npos = fill ? take(8 * B) : 0;
    const size_t o_psess = fill ? take(8 * B) : 0;
    void *scratch = nullptr;
    kvx_status st = pool_alloc(&scratch, off, stream);
    if (st) { delete pl; return st; }
    uint8_t *sb = static_cast<uint8_t *>(scratch);
    MatchScratch m;
    m.push_blocks = reinterpret_cast<int64_t *>(sb + o_push);
    m.sess_start = reinterpret_cast<int64_t *>(sb + o_sess);
    m.pair_src = reinterpret_cast<int64_t *>(sb + o_ps);
    m.pair_dst = reinterpret_cast<int64_t *>(sb + o_pd);
    m.flag = reinterpret_cast<int64_t *>(sb + o_flag);
    m.run_idx = reinterpret_cast<int64_t *>(sb + o_ridx);
    m.run_start = reinterpret_cast<int64_t *>(sb + o_rstart);
    m.tile_count = reinterpret_cast<int64_t *>(sb + o_tcount);
    m.tile_start = reinterpret_cast<int64_t *>(sb + o_tstart);
    m.scan_state = reinterpret_cast<unsigned long long *>(sb + o_state);
    m.scalars = reinterpret_cast<int64_t *>(sb + o_scal);
    m.err = reinterpret_cast<int32_t *>(sb + o_err);
    int32_t *rows = nullptr;   // the plan's run slots (src rows, dst rows, tokens), in its device block
    int64_t *need = fill ? reinterpret_cast<int64_t *>(sb + o_need) : nullptr;
    int64_t *npos = fill ? reinterpret_cast<int64_t *>(sb + o_npos) : nullptr;
    int64_t *pair_sess = fill ? reinterpret_cast<int64_t *>(sb + o_psess) : nullptr;
    if (fill) mf.resident = sb + o_res;

    auto cleanup = [&](kvx_status s) {
        cudaStreamSynchronize(stream);   // nothing may still use the buffers below
        pool_free(scratch);
        if (pl) { if (pl->dev) pool_free(pl->dev); delete pl; }
        return s;
    };
    auto ok = [&](cudaError_t x) { if (x != cudaSuccess && e == cudaSuccess) e = x; };

    ok(cudaMemsetAsync(m.scalars, 0, sizeof(int64_t) * 8 + sizeof(int32_t) * 4 + 8 * 3 * n_state, stream));
    count_launch();
    if (fill) ok(cudaMemsetAsync(mf.resident, 1, (size_t)B, stream));   // unmarked blocks are never pulled
    kvx_match_sessions<<<(unsigned)max(n_sessions, 1), kMatchThreads, 0, stream>>>(tokens, tok_off, n_sessions, block_size,
                                                                        table->view(), remote_hash, rem_off, threshold,
                                                                        mf, out, m.push_blocks, m.sess_start,
                                                                        m.scalars, n_free, m.err);
    ok(cudaGetLastError());

    if (pl && e == cudaSuccess) {
        const std::vector<Pair> pairs = shard_pairs(pl->src, pl->dst);
        EmitShape sh = {};
        sh.src_row_bytes = pl->src.row_bytes();
        sh.dst_row_bytes = pl->dst.row_bytes();
        sh.bs = block_size;
        sh.strided = pl->strided;
        sh.tile_bytes = pl->tile_bytes;
        sh.rows_per_tile = pl->strided ? std::max<int32_t>(1, pl->tile_bytes / pl->width) : 1;
        sh.n_pairs = pl->per_head ? 0 : (int32_t)pairs.size();
        sh.per_head = pl->per_head;
        sh.heads = pl->src.n_shards * pl->src.heads_per_shard;
        sh.hps_s = pl->src.heads_per_shard;
        sh.hps_d = pl->dst.heads_per_shard;
        sh.layout_s = pl->src.layout;
        sh.layout_d = pl->dst.layout;
        sh.head_bytes = pl->src.head_bytes();
        sh.src_pitch = pl->src_pitch;
        sh.dst_pitch = pl->dst_pitch;
        sh.src_head_pitch = pl->src_head_pitch;
        sh.dst_head_pitch = pl->dst_head_pitch;
        // head groups of one block, formed as the host plan builder forms them for a whole block
        sh.heads_per_tile = (int32_t)std::max<int64_t>(1, sh.rows_per_tile / block_size);
        sh.groups = 0;
        for (int32_t g = 0; g < sh.heads; ++sh.groups)
            g += std::min(sh.heads_per_tile, std::min(sh.hps_s - g % sh.hps_s, sh.hps_d - g % sh.hps_d));
        for (size_t q = 0; q < (size_t)sh.n_pairs; ++q) {
            sh.pair_s[q] = pairs[q].s;
            sh.pair_d[q] = pairs[q].d;
            sh.pair_soff[q] = pairs[q].src_seg_off;
            sh.pair_doff[q] = pairs[q].dst_seg_off;
        }
        // a run of L blocks has at most L times the tiles of one block
        const int64_t per_block =
            pl->per_head ? (int64_t)sh.groups * ((block_size + sh.rows_per_tile - 1) / sh.rows_per_tile)
            : (pl->strided ? (block_size + sh.rows_per_tile - 1) / sh.rows_per_tile
                           : ((int64_t)block_size * sh.src_row_bytes + pl->tile_bytes - 1) / pl->tile_bytes) * sh.n_pairs;
        const int64_t tile_cap = B * per_block;
        pl->n_tiles = tile_cap;   // sizes the layout; the real count comes back below
        pl->run_cap = B;
        plan_layout(pl);
        st = pool_alloc(&pl->dev, pl->dev_bytes, stream);
        if (st) return cleanup(st);
        pl->upload_img.assign(pl->off_err - pl->off_src, 0);
        memcpy(pl->upload_img.data(), pl->src_base.data(), sizeof(void *) * pl->src_base.size());
        memcpy(pl->upload_img.data() + (pl->off_dst - pl->off_src), pl->dst_base.data(),
               sizeof(void *) * pl->dst_base.size());
        uint8_t *dev = static_cast<uint8_t *>(pl->dev);
        ok(cudaMemcpyAsync(dev + pl->off_src, pl->upload_img.data(), pl->upload_img.size(), cudaMemcpyHostToDevice,
                           stream));
        ok(cudaMemsetAsync(dev + pl->off_err, 0, sizeof(int32_t) * (size_t)pl->src.n_layers, stream));
        TileDesc *tiles = reinterpret_cast<TileDesc *>(dev + pl->off_tiles);
        rows = reinterpret_cast<int32_t *>(dev + pl->off_runs);

        count_launch(4);
        if (!fill) {
            kvx_emit_pairs<<<grid_for(B, 256), 256, 0, stream>>>(out, m.sess_start, n_sessions, remote_blk, rem_off,
                                                                 free_blocks, &m.scalars[4], m.pair_src, m.pair_dst,
                                                                 m.flag);
        } else {
            count_launch(3);
            kvx_need_flags<<<grid_for(B, 256), 256, 0, stream>>>(out, rem_off, n_sessions, n_pub, mf.resident, need);
            ok(cudaGetLastError());
            ok(exclusive_scan(need, npos, B, nullptr, m.scan_state, &m.scalars[5], m.err, stream));
            kvx_emit_pairs_holes<<<grid_for(B, 256), 256, 0, stream>>>(need, npos, &m.scalars[4], remote_blk, rem_off,
                                                                       n_sessions, n_pub, free_blocks, m.pair_src,
                                                                       m.pair_dst, pair_sess, &m.scalars[5],
                                                                       &m.scalars[0], m.err);
            ok(cudaGetLastError());
            kvx_run_flags<<<grid_for(B, 256), 256, 0, stream>>>(m.pair_src, m.pair_dst, pair_sess, &m.scalars[4],
                                                                m.flag, m.err);
        }
        ok(cudaGetLastError());
        ok(exclusive_scan(m.flag, m.run_idx, B, &m.scalars[4], m.scan_state + n_state, &m.scalars[1], m.err, stream,
                          (mf.flags & KVX_MATCH_TEST_SCAN_STALL) != 0));
        kvx_run_starts<<<grid_for(B, 256), 256, 0, stream>>>(m.flag, m.run_idx, &m.scalars[4], m.run_start, m.err);
        ok(cudaGetLastError());
        kvx_run_tiles<<<grid_for(B, 256), 256, 0, stream>>>(m.run_start, m.scalars, sh, m.tile_count, m.err);
        ok(cudaGetLastError());
        ok(exclusive_scan(m.tile_count, m.tile_start, B, &m.scalars[1], m.scan_state + 2 * n_state, &m.scalars[2],
                          m.err, stream));
        kvx_emit_tiles<<<grid_for(B, 128), 128, 0, stream>>>(m.run_start, m.tile_start, m.scalars, m.pair_src,
                                                             m.pair_dst, sh, tiles, tile_cap, rows, rows + B,
                                                             rows + 2 * B, m.err);
        ok(cudaGetLastError());
    }
    struct { int64_t scal[8]; int32_t err[4]; } back = {};
    ok(cudaMemcpyAsync(&back, m.scalars, sizeof(back), cudaMemcpyDeviceToHost, stream));
    ok(cudaStreamSynchronize(stream));
    const int64_t *h_scal = back.scal;
    const int32_t h_err = back.err[0];
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "kvx_match_prefix"));
    if (h_err & kScanTimedOut) return cleanup(fail(KVX_ETIMEDOUT, "a plan scan waited past its bound for an earlier tile"));
    if (h_err & ~8) return cleanup(fail(KVX_EINVAL, "malformed session or remote offsets (error bits %d)", h_err));
    if (h_err & 8)
        return cleanup(fail(KVX_ENOMEM, "pushing sessions need %lld blocks, free list has %lld", (long long)h_scal[0],
                            (long long)n_free));
    if (pl) {
        // the runs stay on the device (kvx_plan_runs reads them when asked); every pulled block is
        // a whole block, so the tokens per layer are the pulled blocks times the block size
        pl->n_runs_dev = h_scal[1];
        pl->n_tiles = h_scal[2];
        pl->device_tokens = h_scal[4] * block_size;
        finish_plan_shape(pl);
        st = check_pool_memory(pl);
        if (st) return cleanup(st);
        st = event_take(&pl->upload_evt);
        if (st) return cleanup(st);
        e = cudaEventRecord(pl->upload_evt, stream);
        if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaEventRecord(plan)"));
        pl->upload_stream = stream;
        e = cudaGetDevice(&pl->device);
        if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaGetDevice"));
        pl->uploaded = true;
        *out_plan = pl;
        pl = nullptr;
    }
    pool_free(scratch);
    return KVX_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Allocation-free variant of the match decision.
//
// Serving engines usually reserve nearly all free HBM for their paged KV pools at start-up and
// allow no device allocation on the request path afterwards: a cudaMalloc there can fail once the
// pools are carved out, and cudaMalloc / cudaFree may synchronise the device and stall every other
// stream. kvx_match_prefix_static serves such callers. Its scratch (per-session pushed-block
// counts, their exclusive scan, totals and error bits) is the file-scope array below, sized for
// at most kStaticMaxSessions sessions per call (about 1 MiB, held by every GPU
// that loads the library until the process exits).
// ------------------------------------------------------------------------------------------------

namespace kvx {

constexpr int32_t kStaticMaxSessions = 65536;
constexpr size_t kStaticPushOff = 0;
constexpr size_t kStaticSessOff = kStaticPushOff + sizeof(int64_t) * kStaticMaxSessions;
constexpr size_t kStaticScalOff = kStaticSessOff + sizeof(int64_t) * kStaticMaxSessions;
constexpr size_t kStaticErrOff = kStaticScalOff + sizeof(int64_t) * 8;   // right after the scalars
constexpr size_t kStaticBytes = kStaticErrOff + sizeof(int32_t) * 4;

static __device__ __align__(256) unsigned char g_match_scratch[kStaticBytes];

// In host code g_match_scratch names a host-side stand-in, not device memory: the device address
// is looked up once per device (with that device current) and cached. The cache lives as long as
// the device's primary context; like the library's other per-device state (lanes, memory pool,
// events) it does not survive a device reset, which the header states.
static std::mutex g_static_mu;
static std::map<int, unsigned char *> g_static_addr;

static kvx_status static_scratch(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_static_mu);
    auto it = g_static_addr.find(dev);
    if (it == g_static_addr.end()) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_match_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(match scratch)");
        it = g_static_addr.emplace(dev, static_cast<unsigned char *>(p)).first;
    }
    *out = it->second;
    return KVX_OK;
}

}  // namespace kvx

extern "C" kvx_status kvx_match_prefix_static(const uint32_t *tokens, const int64_t *tok_off, int32_t n_sessions,
                                              int32_t block_size, kvx_table_t table, const uint64_t *remote_hash,
                                              const int64_t *rem_off, int32_t threshold, int64_t n_free,
                                              kvx_match_result *out, cudaStream_t stream) {
    if (n_sessions < 0 || block_size < 1 || n_free < 0) return fail(KVX_EINVAL, "bad counts");
    if (n_sessions > kStaticMaxSessions)
        return fail(KVX_EINVAL, "kvx_match_prefix_static takes at most %d sessions per call (got %d); its scratch "
                                "is a fixed array", kStaticMaxSessions, n_sessions);
    if (!table) return fail(KVX_EINVAL, "NULL table");
    if (n_sessions == 0) return KVX_OK;
    if (!tokens || !tok_off || !rem_off || !remote_hash || !out) return fail(KVX_EINVAL, "NULL device array");
    unsigned char *sc = nullptr;
    kvx_status st = static_scratch(&sc);
    if (st) return st;
    int64_t *push_blocks = reinterpret_cast<int64_t *>(sc + kStaticPushOff);
    int64_t *sess_start = reinterpret_cast<int64_t *>(sc + kStaticSessOff);
    int64_t *scalars = reinterpret_cast<int64_t *>(sc + kStaticScalOff);
    int32_t *err = reinterpret_cast<int32_t *>(sc + kStaticErrOff);

    // the kernels bound their reads by the two CSR totals themselves (no host round trip); the
    // array keeps the previous call's contents: the totals and error bits must start at zero
    cudaError_t e = cudaMemsetAsync(scalars, 0, sizeof(int64_t) * 8 + sizeof(int32_t) * 4, stream);
    if (e == cudaSuccess) {
        count_launch();
        kvx_match_sessions<<<(unsigned)max(n_sessions, 1), kMatchThreads, 0, stream>>>(tokens, tok_off, n_sessions, block_size,
                                                                            table->view(), remote_hash, rem_off, threshold,
                                                                            MatchFlags{0, nullptr, 0, nullptr}, out,
                                                                            push_blocks, sess_start, scalars, n_free,
                                                                            err);
        e = cudaGetLastError();
    }
    struct { int64_t scal[8]; int32_t err[4]; } back = {};
    if (e == cudaSuccess) e = cudaMemcpyAsync(&back, scalars, sizeof(back), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    const int64_t need = back.scal[0];
    const int32_t h_err = back.err[0];
    if (e != cudaSuccess) return cuda_fail(e, "kvx_match_prefix_static");
    if (h_err & ~8) return fail(KVX_EINVAL, "malformed session or remote offsets (error bits %d)", h_err);
    if (h_err & 8)
        return fail(KVX_ENOMEM, "pushing sessions need %lld blocks, free list has %lld", (long long)need,
                    (long long)n_free);
    return KVX_OK;
}
