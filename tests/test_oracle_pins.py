"""Pins of the oracle against things other than itself (CPU only).

- FNV-1a: the hash authors' published test vectors (tests/golden/fnv1a64_vectors.txt).
- Block hashes: the message encoding rebuilt in Python bytes and hashed with the pinned FNV; chain
  sensitivity; shared prefixes hash alike.
- Push: numpy tensor-view route, consumer-side per-byte brute force, one-memcpy special case,
  canaries, producer unchanged, write-once markers.
- Runs: hand-worked examples, sum / maximality / round-trip invariants.
- Match: a naive per-block Python loop, threshold edges, degenerate sessions, free-list exhaustion.
"""
import os
import zlib

import numpy as np
import pytest

import kvx_inputs
import oracle
from helpers import ceil_div, dst_side_map, host_pool, numpy_route_push, random_requests

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PoolGeom = kvx_inputs.PoolGeom


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def read_fnv_vectors():
    out = []
    with open(os.path.join(GOLDEN, "fnv1a64_vectors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            q2 = line.rindex('"')
            out.append((line[1:q2].encode("ascii"), int(line[q2 + 1:].strip(), 16)))
    return out


# ---------------------------------------------------------------------------------------------
# FNV-1a and block hashes
# ---------------------------------------------------------------------------------------------

def test_fnv_published_vectors(orc):
    vecs = read_fnv_vectors()
    assert len(vecs) >= 5
    for data, want in vecs:
        assert orc.fnv1a64(data) == want, data
    assert orc.offset_basis() == dict(vecs)[b""]


def test_fnv_continues_from_state(orc):
    a, b = b"prefill->", b"decode"
    assert orc.fnv1a64(a + b) == orc.fnv1a64(b, orc.fnv1a64(a))


@pytest.mark.parametrize("block_size,n_tokens", [(64, 64 * 5 + 17), (4, 9), (1, 7), (64, 63), (64, 0)])
def test_block_hash_encoding(orc, block_size, n_tokens):
    rng = np.random.default_rng(11)
    toks = rng.integers(0, 2**32, n_tokens, dtype=np.uint64).astype(np.uint32)
    got = orc.block_hashes(toks, block_size)
    assert len(got) == n_tokens // block_size          # a trailing partial block is not hashed
    parent = 0
    for j in range(n_tokens // block_size):
        msg = parent.to_bytes(8, "little") + toks[j * block_size:(j + 1) * block_size].astype("<u4").tobytes()
        want = orc.fnv1a64(msg)
        assert int(got[j]) == want
        parent = want


def test_block_hash_first_block_parent_zero(orc):
    toks = np.arange(64, dtype=np.uint32)
    msg = bytes(8) + toks.astype("<u4").tobytes()
    assert int(orc.block_hashes(toks, 64)[0]) == orc.fnv1a64(msg)
    # token ids are little endian: token 1 contributes octets 01 00 00 00
    assert msg[8 + 4:8 + 8] == b"\x01\x00\x00\x00"


def test_block_hash_chain_sensitivity(orc):
    rng = np.random.default_rng(3)
    toks = rng.integers(0, kvx_inputs.VOCAB, 64 * 12, dtype=np.int64).astype(np.uint32)
    base = orc.block_hashes(toks, 64)
    for j in (0, 5, 11):
        t2 = toks.copy()
        t2[j * 64 + 13] ^= 1
        h2 = orc.block_hashes(t2, 64)
        assert np.array_equal(h2[:j], base[:j])
        assert np.all(h2[j:] != base[j:])


def test_shared_system_prompt_hashes_alike(orc):
    w = kvx_inputs.bidir_mla_fp8(seed=5, n_sessions=3, n_layers=1, hist_range=(100, 300))
    hs = [orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], 64) for s in range(3)]
    for s in (1, 2):
        assert np.array_equal(hs[s][:16], hs[0][:16])   # 1024 shared tokens = 16 blocks
        assert hs[s][16] != hs[0][16]


# ---------------------------------------------------------------------------------------------
# Push
# ---------------------------------------------------------------------------------------------

GEOMS = {
    # name: (src geometry, dst geometry)
    "equal": (PoolGeom(2, 2, 1, 2, 4, 2, 4, 12), PoolGeom(2, 2, 1, 2, 4, 2, 4, 12)),
    "merge4to1_bs4to8": (PoolGeom(1, 2, 4, 1, 2, 2, 4, 10), PoolGeom(1, 2, 1, 4, 2, 2, 8, 6)),
    "split1to2_bs8to2": (PoolGeom(1, 1, 1, 4, 2, 2, 8, 5), PoolGeom(1, 1, 2, 2, 2, 2, 2, 20)),
    "bs1": (PoolGeom(1, 2, 1, 2, 2, 1, 1, 24), PoolGeom(1, 2, 1, 2, 2, 1, 1, 24)),
    "odd_head_bytes": (PoolGeom(1, 1, 2, 1, 3, 1, 3, 9), PoolGeom(1, 1, 1, 2, 3, 1, 5, 7)),
    "mla_like": (PoolGeom(2, 1, 1, 1, 6, 1, 4, 8), PoolGeom(2, 1, 1, 1, 6, 1, 4, 8)),
    "hnd_equal": (PoolGeom(1, 2, 1, 3, 4, 2, 4, 10, 1), PoolGeom(1, 2, 1, 3, 4, 2, 4, 10, 1)),
    "nhd_to_hnd_bs4to8": (PoolGeom(1, 1, 2, 2, 4, 2, 4, 10), PoolGeom(1, 1, 1, 4, 4, 2, 8, 6, 1)),
    "hnd_to_nhd_split": (PoolGeom(1, 2, 1, 4, 2, 2, 8, 5, 1), PoolGeom(1, 2, 2, 2, 2, 2, 4, 10)),
}


@pytest.mark.parametrize("name", sorted(GEOMS))
def test_push_matches_numpy_route_and_dst_side_map(orc, name):
    sg, dg = GEOMS[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    max_tok = min(sg.n_blocks * sg.block_size, dg.n_blocks * dg.block_size) // 3
    for trial in range(3):
        reqs = random_requests(rng, sg, dg, 3, max_tok)
        src = host_pool(sg, 7 + trial)
        dst = host_pool(dg, 0, fill=0xA5)
        src_copy = [b.copy() for b in src]
        want_np = numpy_route_push(sg, src, dg, dst, reqs)
        want_map = dst_side_map(sg, src, dg, dst, reqs)
        orc.push(sg, src, dg, dst, reqs)
        for a, b, c in zip(dst, want_np, want_map):
            assert np.array_equal(a, b)
            assert np.array_equal(a, c)
        for a, b in zip(src, src_copy):
            assert np.array_equal(a, b)              # producer pool is never written


def test_push_all_contiguous_is_one_memcpy(orc):
    g = PoolGeom(1, 1, 1, 2, 8, 2, 4, 16)
    src = host_pool(g, 3)
    dst = host_pool(g, 0, fill=0)
    n_blocks, off = 6, 9
    orc.push(g, src, g, dst, [(n_blocks * 4, np.arange(n_blocks), np.arange(off, off + n_blocks))])
    bb = g.block_size * g.row_bytes
    assert np.array_equal(dst[0][off * bb:(off + n_blocks) * bb], src[0][:n_blocks * bb])
    assert not dst[0][:off * bb].any() and not dst[0][(off + n_blocks) * bb:].any()


def test_push_partial_last_block_keeps_canary(orc):
    g = PoolGeom(1, 1, 1, 1, 4, 2, 8, 4)
    src = host_pool(g, 4)
    dst = host_pool(g, 0, fill=0xAD)
    orc.push(g, src, g, dst, [(11, np.array([0, 1]), np.array([3, 1]))])
    rb = g.row_bytes
    assert np.array_equal(dst[0][3 * 8 * rb:4 * 8 * rb], src[0][:8 * rb])
    assert np.array_equal(dst[0][1 * 8 * rb:(8 + 3) * rb], src[0][8 * rb:11 * rb])
    assert np.all(dst[0][(8 + 3) * rb:16 * rb] == 0xAD)   # slots 3..7 of the last block
    assert np.all(dst[0][:8 * rb] == 0xAD) and np.all(dst[0][16 * rb:24 * rb] == 0xAD)


def test_push_write_once_markers(orc):
    """Every producer head slot carries a unique 8-byte marker; after the push, the consumer slots
    that changed hold pairwise-distinct markers, as many as tokens x heads x layers x planes."""
    sg, dg = GEOMS["merge4to1_bs4to8"]
    sg = sg.replace(head_dim=4)                       # 8-byte heads hold one uint64 marker
    dg = dg.replace(head_dim=4)
    src = []
    for i in range(sg.n_buffers):
        n = sg.buffer_bytes // 8
        src.append((np.arange(n, dtype=np.uint64) + np.uint64(i << 32) + np.uint64(1)).view(np.uint8))
    dst = host_pool(dg, 0, fill=0)
    reqs = [(13, np.array([4, 0, 7, 2]), np.array([5, 2])), (5, np.array([9, 8]), np.array([0]))]
    orc.push(sg, src, dg, dst, reqs)
    vals = np.concatenate([b.view(np.uint64) for b in dst])
    written = vals[vals != 0]
    heads = sg.n_shards * sg.heads_per_shard
    assert len(written) == (13 + 5) * heads * sg.n_layers * sg.n_planes
    assert len(np.unique(written)) == len(written)


def test_push_rejects_out_of_range(orc):
    g = PoolGeom(1, 1, 1, 1, 2, 1, 2, 4)
    with pytest.raises(ValueError):
        orc.push(g, host_pool(g, 1), g, host_pool(g, 0, 0), [(4, np.array([0, 4]), np.array([0, 1]))])


# ---------------------------------------------------------------------------------------------
# Runs
# ---------------------------------------------------------------------------------------------

HAND_RUNS = [
    # (src ids, dst ids, expected [(src, dst, len), ...]) worked by hand from the merge rule
    ([0, 1, 2, 3], [10, 11, 12, 13], [(0, 10, 4)]),
    ([0, 1, 2, 3], [10, 12, 14, 16], [(0, 10, 1), (1, 12, 1), (2, 14, 1), (3, 16, 1)]),
    ([5, 6, 9, 10], [1, 2, 3, 4], [(5, 1, 2), (9, 3, 2)]),          # breaks on src only
    ([0, 1, 2, 3], [7, 8, 3, 4], [(0, 7, 2), (2, 3, 2)]),           # breaks on dst only
    ([3, 2, 1], [0, 1, 2], [(3, 0, 1), (2, 1, 1), (1, 2, 1)]),      # descending is not contiguous
    ([], [], []),
    ([42], [7], [(42, 7, 1)]),
]


@pytest.mark.parametrize("src,dst,want", HAND_RUNS)
def test_block_runs_hand_examples(orc, src, dst, want):
    rs, rd, rl = orc.block_runs(src, dst)
    assert list(zip(rs.tolist(), rd.tolist(), rl.tolist())) == want


def test_token_runs_hand_example(orc):
    # bs_src 2, bs_dst 4, 7 tokens. src rows: 10 11 12 13 0 1 2; dst rows: 8 9 10 11 36 37 38.
    rs, rd, rl = orc.token_runs(7, 2, [5, 6, 0, 1], 4, [2, 9])
    assert list(zip(rs.tolist(), rd.tolist(), rl.tolist())) == [(10, 8, 4), (0, 36, 3)]


def test_runs_invariants_random(orc):
    rng = np.random.default_rng(9)
    for _ in range(50):
        n = int(rng.integers(0, 200))
        src = kvx_inputs.chunked_order(rng, 300, mean=2.0)[:n]
        dst = kvx_inputs.chunked_order(rng, 300, p_single=0.8, mean_multi=4.0)[:n]
        rs, rd, rl = orc.block_runs(src, dst)
        assert rl.sum() == n and np.all(rl >= 1)
        for k in range(len(rs) - 1):                  # maximal: no two neighbours could merge
            assert not (rs[k] + rl[k] == rs[k + 1] and rd[k] + rl[k] == rd[k + 1])
        es = np.concatenate([np.arange(a, a + c) for a, c in zip(rs, rl)]) if n else np.zeros(0)
        ed = np.concatenate([np.arange(a, a + c) for a, c in zip(rd, rl)]) if n else np.zeros(0)
        assert np.array_equal(es, src) and np.array_equal(ed, dst)   # round trip
        # with equal block sizes, token runs are the block runs in rows, last one cut at n_tokens
        bs = 16
        n_tok = max(0, n * bs - int(rng.integers(0, bs)))
        nb = ceil_div(n_tok, bs)
        ts, td, tl = orc.token_runs(n_tok, bs, src, bs, dst)
        bs_s, bd_s, bl_s = orc.block_runs(src[:nb], dst[:nb])
        assert np.array_equal(ts, bs_s.astype(np.int64) * bs) and np.array_equal(td, bd_s.astype(np.int64) * bs)
        assert tl.sum() == n_tok


# ---------------------------------------------------------------------------------------------
# Match
# ---------------------------------------------------------------------------------------------

def naive_match(orc, tokens, tok_off, bs, local_keys, remote_hash, remote_blk, rem_off, threshold, free,
                fill_holes=False, keep_last=False, expiry=None, now=0):
    keys = set(int(k) for k in local_keys)
    res = dict(local_hit=[], remote_hit=[], missing=[], push=[])
    pulled = []
    for s in range(len(tok_off) - 1):
        h = [int(x) for x in orc.block_hashes(tokens[tok_off[s]:tok_off[s + 1]], bs)]
        rem = [int(x) for x in remote_hash[rem_off[s]:rem_off[s + 1]]]
        if expiry is not None and now >= expiry[s]:
            rem = []
        loc = 0
        while loc < len(h) and h[loc] in keys:
            loc += 1
        rh = 0
        while rh < len(h) and rh < len(rem) and h[rh] == rem[rh]:
            rh += 1
        if keep_last and rh > 0 and rh * bs >= tok_off[s + 1] - tok_off[s]:
            rh -= 1
        if fill_holes:
            take = [j for j in range(rh) if h[j] not in keys]
        else:
            take = list(range(loc, rh))
        miss = len(take) * bs
        res["local_hit"].append(loc)
        res["remote_hit"].append(rh)
        res["missing"].append(miss)
        res["push"].append(int(miss > 0 and miss >= threshold))
        pulled.append(take)
    pairs_s, pairs_d, cur = [], [], 0
    for s in range(len(tok_off) - 1):
        if res["push"][s]:
            for i, j in enumerate(pulled[s]):
                pairs_s.append(int(remote_blk[rem_off[s] + j]))
                pairs_d.append(int(free[cur + i]))
            cur += len(pulled[s])
    return res, pairs_s, pairs_d


def test_match_equals_naive_loop(orc):
    w = kvx_inputs.bidir_mla_fp8(seed=21, n_sessions=12, n_layers=1, system_tokens=256,
                                 hist_range=(64, 2000), resident_p=0.7, threshold=128)
    hashes = [orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], 64) for s in range(w.n_sessions)]
    allh = np.concatenate(hashes)
    remote = allh.copy()
    rng = np.random.default_rng(2)
    flip = rng.random(len(remote)) < 0.02               # some published hashes disagree
    remote[flip] ^= np.uint64(1)
    keys = np.unique(allh[w.resident])
    got = orc.match(w.tokens, w.tok_off, 64, keys, remote, w.remote_blk, w.rem_off, w.threshold, w.free_blocks)
    want, ps, pd = naive_match(orc, w.tokens, w.tok_off, 64, keys, remote, w.remote_blk, w.rem_off,
                               w.threshold, w.free_blocks)
    for k in ("local_hit", "remote_hit", "missing", "push"):
        assert got[k].tolist() == want[k], k
    assert got["pair_src"].tolist() == ps and got["pair_dst"].tolist() == pd
    assert got["status"] == 0 and sum(want["push"]) > 0


def _session_case(orc, bs, n_blocks, l_loc, l_rem, extra_resident=()):
    rng = np.random.default_rng(100 + n_blocks + l_loc + l_rem)
    toks = rng.integers(0, kvx_inputs.VOCAB, n_blocks * bs, dtype=np.int64).astype(np.uint32)
    h = orc.block_hashes(toks, bs)
    keys = np.concatenate([h[:l_loc], h[list(extra_resident)]]) if len(extra_resident) else h[:l_loc]
    remote = h.copy()
    if l_rem < n_blocks:
        remote[l_rem] ^= np.uint64(0x5A)
    return toks, keys, remote


@pytest.mark.parametrize("l_rem,want_push", [(511, 0), (512, 1), (513, 1)])
def test_match_threshold_edges_tokens(orc, l_rem, want_push):
    bs, n = 1, 600
    toks, keys, remote = _session_case(orc, bs, n, 0, l_rem)
    got = orc.match(toks, [0, n], bs, keys, remote, np.arange(n), [0, n], 512, np.arange(n))
    assert got["missing"].tolist() == [l_rem] and got["push"].tolist() == [want_push]


@pytest.mark.parametrize("l_rem,want_push", [(7, 0), (8, 1), (9, 1)])
def test_match_threshold_edges_blocks(orc, l_rem, want_push):
    bs, n = 64, 12                                     # missing = 448, 512, 576 tokens
    toks, keys, remote = _session_case(orc, bs, n, 0, l_rem)
    got = orc.match(toks, [0, n * bs], bs, keys, remote, np.arange(n), [0, n], 512, np.arange(n))
    assert got["missing"].tolist() == [l_rem * 64] and got["push"].tolist() == [want_push]


def test_match_degenerate_sessions(orc):
    bs, n = 4, 10
    cases = [
        # (l_loc, l_rem, extra resident blocks, published count, want (local, remote, missing, push))
        (6, 4, (), n, (6, 4, 0, 0)),          # remote span inside the local hit: nothing to pull
        (n, n, (), n, (n, n, 0, 0)),          # full local hit
        (2, n, (), 0, (2, 0, 0, 0)),          # empty published list
        (2, n, (5, 6), n, (2, n, 32, 1)),     # resident blocks past the first miss are not reused
        (0, 3, (), 2, (0, 2, 8, 1)),          # published list shorter than the session
    ]
    for l_loc, l_rem, extra, n_pub, want in cases:
        toks, keys, remote = _session_case(orc, bs, n, l_loc, l_rem, extra)
        got = orc.match(toks, [0, n * bs], bs, keys, remote[:n_pub], np.arange(n_pub), [0, n_pub], 1,
                        np.arange(100))
        assert (got["local_hit"][0], got["remote_hit"][0], got["missing"][0], got["push"][0]) == want


def test_match_free_list_order_and_exhaustion(orc):
    bs, n = 2, 6
    parts, keys_all, rem_all = [], [], []
    for s in range(3):
        toks, keys, remote = _session_case(orc, bs, n, s, n)
        parts.append(toks)
        keys_all.append(keys)
        rem_all.append(remote)
    tokens = np.concatenate(parts)
    tok_off = [0, n * bs, 2 * n * bs, 3 * n * bs]
    rem_off = [0, n, 2 * n, 3 * n]
    keys = np.concatenate(keys_all)
    remote = np.concatenate(rem_all)
    rblk = np.arange(100, 100 + 3 * n)
    free = np.array([50, 51, 52, 40, 41, 42, 43, 44, 45, 46, 47, 48, 49, 30, 31])   # 6 + 5 + 4 = 15 needed
    got = orc.match(tokens, tok_off, bs, keys, remote, rblk, rem_off, 1, free)
    assert got["status"] == 0
    assert got["dst_start"].tolist() == [0, 6, 11]
    assert got["pair_src"].tolist() == list(range(100, 106)) + list(range(107, 112)) + list(range(114, 118))
    assert got["pair_dst"].tolist() == free.tolist()
    short = orc.match(tokens, tok_off, bs, keys, remote, rblk, rem_off, 1, free[:14])
    assert short["status"] == 5 and len(short["pair_src"]) == 0
    assert short["push"].tolist() == [1, 1, 1]


@pytest.mark.parametrize("fill_holes,keep_last,ttl", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 1)])
def test_match_options_equal_naive_loop(orc, fill_holes, keep_last, ttl):
    w = kvx_inputs.bidir_mla_fp8(seed=40 + fill_holes + 2 * keep_last + 4 * ttl, n_sessions=14, n_layers=1,
                                 system_tokens=256, hist_range=(0, 1500), resident_p=0.5, threshold=128)
    # some sessions end exactly on a block boundary so that keep_last bites
    hashes = [orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], 64) for s in range(w.n_sessions)]
    allh = np.concatenate(hashes)
    keys = np.unique(allh[w.resident])
    expiry = np.random.default_rng(7).integers(0, 200, w.n_sessions) if ttl else None
    flags = (orc.FILL_HOLES if fill_holes else 0) | (orc.KEEP_LAST if keep_last else 0)
    got = orc.match(w.tokens, w.tok_off, 64, keys, allh, w.remote_blk, w.rem_off, w.threshold, w.free_blocks,
                    flags=flags, expiry=expiry, now=100)
    want, ps, pd = naive_match(orc, w.tokens, w.tok_off, 64, keys, allh, w.remote_blk, w.rem_off, w.threshold,
                               w.free_blocks, fill_holes=bool(fill_holes), keep_last=bool(keep_last),
                               expiry=expiry, now=100)
    for k in ("local_hit", "remote_hit", "missing", "push"):
        assert got[k].tolist() == want[k], k
    assert got["pair_src"].tolist() == ps and got["pair_dst"].tolist() == pd


def test_match_options_hand_cases(orc):
    bs, n = 4, 8
    toks, keys, remote = _session_case(orc, bs, n, 2, n, extra_resident=(4, 6))
    args = (toks, [0, n * bs], bs, keys, remote, np.arange(10, 10 + n), [0, n], 1, np.arange(50, 60))
    plain = orc.match(*args)
    assert (plain["local_hit"][0], plain["remote_hit"][0], plain["missing"][0]) == (2, 8, 24)
    assert plain["pair_src"].tolist() == [12, 13, 14, 15, 16, 17]
    holes = orc.match(*args, flags=orc.FILL_HOLES)            # blocks 4 and 6 are reused in place
    assert holes["missing"][0] == 16 and holes["pair_src"].tolist() == [12, 13, 15, 17]
    assert holes["pair_dst"].tolist() == [50, 51, 52, 53]
    last = orc.match(*args, flags=orc.KEEP_LAST)               # 32 tokens, all covered: last block recomputed
    assert last["remote_hit"][0] == 7 and last["missing"][0] == 20
    both = orc.match(*args, flags=orc.FILL_HOLES | orc.KEEP_LAST)
    assert both["pair_src"].tolist() == [12, 13, 15]
    expired = orc.match(*args, expiry=np.array([100]), now=100)
    assert expired["remote_hit"][0] == 0 and expired["push"][0] == 0
    alive = orc.match(*args, expiry=np.array([101]), now=100)
    assert alive["remote_hit"][0] == 8
    partial = orc.match(toks[:-1], [0, n * bs - 1], bs, keys, remote[:n - 1], np.arange(n - 1), [0, n - 1], 1,
                        np.arange(9), flags=orc.KEEP_LAST)     # a partial last block is computed anyway
    assert partial["remote_hit"][0] == 7
