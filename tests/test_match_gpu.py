"""GPU parity of the bidirectional reuse path through the C-ABI: block hashes, the resident table, the
per-session match decision, the device-built decode->prefill plan and its push, all against the
oracle (integer work: bit-exact)."""
import numpy as np
import pytest

import kvx_inputs
import oracle
from gpu_helpers import canary_host, check_layers, device_pool

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
kvx = pytest.importorskip("disaggregated_prefill_decode_gb300.kvx")

PoolGeom = kvx_inputs.PoolGeom


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


def dev(a, dtype):
    """numpy -> device tensor with the same bits (uint32 / uint64 travel as int32 / int64)."""
    a = np.ascontiguousarray(a)
    view = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
    if len(a) == 0:
        a = np.zeros(1, a.dtype)
    return torch.from_numpy(a.view(view)).to("cuda")


def results(out_t, n):
    return out_t.cpu().numpy().view(kvx.MATCH_RESULT_DTYPE)[:n]


# ---------------------------------------------------------------------------------------------
# hashes and table
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [64, 4, 1])
def test_block_hashes_match_oracle(bs):
    rng = np.random.default_rng(bs)
    lens = [0, 1, bs - 1, bs, 5 * bs + 3, 700, 2 * bs]
    toks = [rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32) for n in lens]
    tok_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    nh = [n // bs for n in lens]
    hash_off = np.concatenate([[0], np.cumsum(nh)]).astype(np.int64)
    out = torch.zeros(max(int(hash_off[-1]), 1), dtype=torch.int64, device="cuda")
    kvx.kvx_block_hashes(dev(np.concatenate(toks), np.uint32), dev(tok_off, np.int64), len(lens), bs, out,
                         dev(hash_off, np.int64))
    got = out.cpu().numpy().view(np.uint64)
    orc = oracle.load()
    for s, t in enumerate(toks):
        assert np.array_equal(got[hash_off[s]:hash_off[s + 1]], orc.block_hashes(t, bs)), s


def test_block_hashes_continue_from_a_parent():
    """A turn's new blocks hashed from the hash of the block before them equal the tail of the whole
    stream's chain: each session split at a random block boundary (empty halves included)."""
    rng = np.random.default_rng(7)
    bs, n = 64, 20
    lens = rng.integers(0, 60, n) * bs + rng.integers(0, bs, n)
    streams = [rng.integers(0, 151936, int(l)).astype(np.uint32) for l in lens]
    orc = oracle.load()
    full = [orc.block_hashes(t, bs) for t in streams]
    cut = [int(rng.integers(0, len(h) + 1)) for h in full]                  # in blocks
    head = [t[:k * bs] for t, k in zip(streams, cut)]
    tail = [t[k * bs:] for t, k in zip(streams, cut)]
    parent = np.array([h[k - 1] if k > 0 else 0 for h, k in zip(full, cut)], dtype=np.uint64)

    def hashes(parts, par):
        tok = np.concatenate(parts).astype(np.uint32) if parts else np.zeros(0, np.uint32)
        off = np.concatenate([[0], np.cumsum([len(p) for p in parts])]).astype(np.int64)
        hoff = np.concatenate([[0], np.cumsum([len(p) // bs for p in parts])]).astype(np.int64)
        out = torch.zeros(max(int(hoff[-1]), 1), dtype=torch.int64, device="cuda")
        kvx.kvx_block_hashes_ex(dev(tok, np.uint32), dev(off, np.int64), len(parts), bs,
                                None if par is None else dev(par, np.uint64), out, dev(hoff, np.int64))
        got = out.cpu().numpy().view(np.uint64)
        return [got[hoff[i]:hoff[i + 1]] for i in range(len(parts))]

    first, second = hashes(head, None), hashes(tail, parent)
    for i in range(n):
        assert np.array_equal(np.concatenate([first[i], second[i]]), full[i]), i


def test_block_hashes_reject_short_output_range():
    tok_off = dev(np.array([0, 128], np.int64), np.int64)
    hash_off = dev(np.array([0, 1], np.int64), np.int64)       # 2 full blocks, room for 1
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(kvx.KvxError) as ei:
        kvx.kvx_block_hashes(dev(np.zeros(128, np.uint32), np.uint32), tok_off, 1, 64, out, hash_off)
    assert ei.value.status == kvx.KVX_ERANGE


def test_table_build_and_lookup():
    rng = np.random.default_rng(5)
    keys = np.unique(rng.integers(1, 2**63, 5000, dtype=np.int64).astype(np.uint64))
    keys = np.concatenate([keys, np.array([0], np.uint64)])      # key 0 is a legal hash
    vals = rng.integers(0, 10**6, len(keys)).astype(np.int32)
    table = kvx.kvx_table_build(dev(keys, np.uint64), dev(vals, np.int32), len(keys))
    probe = np.concatenate([keys, rng.integers(1, 2**63, 3000, dtype=np.int64).astype(np.uint64)])
    out = torch.empty(len(probe), dtype=torch.int32, device="cuda")
    kvx.kvx_table_lookup(table, dev(probe, np.uint64), len(probe), out)
    got = out.cpu().numpy()
    want = dict(zip(keys.tolist(), vals.tolist()))
    assert got.tolist() == [want.get(k, -1) for k in probe.tolist()]
    kvx.kvx_table_destroy(table)
    with pytest.raises(kvx.KvxError) as ei:
        kvx.kvx_table_build(dev(np.array([7, 9, 7], np.uint64), np.uint64), dev(np.arange(3, dtype=np.int32), np.int32), 3)
    assert ei.value.status == kvx.KVX_EINVAL
    empty = kvx.kvx_table_build(None, None, 0)
    kvx.kvx_table_lookup(empty, dev(keys[:10], np.uint64), 10, out)
    assert out[:10].cpu().tolist() == [-1] * 10
    kvx.kvx_table_destroy(empty)


# ---------------------------------------------------------------------------------------------
# match + device-built plan + push
# ---------------------------------------------------------------------------------------------

class Case:
    """A bidirectional workload on the device: published hashes and resident keys from the oracle."""

    def __init__(self, w, flip_frac=0.0, seed=0):
        orc = oracle.load()
        self.w = w
        hs = [orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], w.block_size) for s in range(w.n_sessions)]
        allh = np.concatenate(hs) if hs else np.zeros(0, np.uint64)
        self.remote_hash = allh.copy()
        if flip_frac:
            flip = np.random.default_rng(seed).random(len(allh)) < flip_frac
            self.remote_hash[flip] ^= np.uint64(1)
        self.keys = np.unique(allh[w.resident])
        self.t_tokens = dev(w.tokens, np.uint32)
        self.t_tok_off = dev(w.tok_off, np.int64)
        self.t_rh = dev(self.remote_hash, np.uint64)
        self.t_rb = dev(w.remote_blk, np.int32)
        self.t_ro = dev(w.rem_off, np.int64)
        self.t_free = dev(w.free_blocks, np.int32)
        self.table = kvx.kvx_table_build(dev(self.keys, np.uint64), dev(np.arange(len(self.keys), dtype=np.int32),
                                                                        np.int32), len(self.keys))

    def oracle_match(self, n_free=None, flags=0, expiry=None, now=0):
        w = self.w
        free = w.free_blocks if n_free is None else w.free_blocks[:n_free]
        return oracle.load().match(w.tokens, w.tok_off, w.block_size, self.keys, self.remote_hash, w.remote_blk,
                                   w.rem_off, w.threshold, free, flags=flags, expiry=expiry, now=now)

    def match(self, remote_pool=None, local_pool=None, n_free=None, want_plan=True, flags=0, expiry=None, now=0):
        w = self.w
        out = torch.zeros(max(w.n_sessions, 1) * 24, dtype=torch.uint8, device="cuda")
        nf = len(w.free_blocks) if n_free is None else n_free
        st, plan = kvx.kvx_match_prefix(self.t_tokens, self.t_tok_off, w.n_sessions, w.block_size, self.table, self.t_rh,
                                        self.t_rb, self.t_ro, w.threshold, self.t_free, nf, remote_pool, local_pool, out,
                                        want_plan=want_plan, flags=flags,
                                        expiry=None if expiry is None else dev(expiry, np.int64), now=now)
        return st, plan, results(out, w.n_sessions)

    def close(self):
        kvx.kvx_table_destroy(self.table)


def assert_decisions(got, want):
    assert got["local_hit_blocks"].tolist() == want["local_hit"].tolist()
    assert got["remote_hit_blocks"].tolist() == want["remote_hit"].tolist()
    assert got["missing_tokens"].tolist() == want["missing"].tolist()
    assert got["push"].tolist() == want["push"].tolist()
    assert got["dst_start"].tolist() == want["dst_start"].tolist()


def trim_to_blocks(w, sessions):
    """Cut the given sessions' token streams to whole blocks (their published blocks are unchanged)."""
    parts, offs = [], [0]
    for s in range(w.n_sessions):
        t = w.tokens[w.tok_off[s]:w.tok_off[s + 1]]
        if s in sessions:
            t = t[:len(t) // w.block_size * w.block_size]
        parts.append(t)
        offs.append(offs[-1] + len(t))
    w.tokens = np.concatenate(parts).astype(np.uint32)
    w.tok_off = np.asarray(offs, np.int64)


def oracle_requests(c, want):
    """The pushes the oracle's match implies: one request per pushing session (its pulled blocks in
    order; with hole filling they need not be consecutive session blocks, which a copy ignores)."""
    w, reqs, k = c.w, [], 0
    for s in range(w.n_sessions):
        if want["push"][s]:
            nb = int(want["missing"][s]) // w.block_size
            reqs.append((nb * w.block_size, want["pair_src"][k:k + nb], want["pair_dst"][k:k + nb]))
            k += nb
    return reqs


def test_match_decisions_and_plan_runs_reduced():
    w = kvx_inputs.bidir_mla_fp8(seed=21, n_sessions=24, n_layers=2, system_tokens=256, hist_range=(64, 3000),
                                 resident_p=0.6, threshold=256)
    c = Case(w, flip_frac=0.01, seed=3)
    want = c.oracle_match()
    assert want["status"] == 0 and want["push"].sum() > 3 and (want["push"] == 0).sum() > 0
    st, plan, got = c.match(want_plan=False)
    assert st == kvx.KVX_OK and plan is None
    assert_decisions(got, want)
    c.close()


@pytest.mark.parametrize("flags", [0, kvx.KVX_MATCH_FILL_HOLES, kvx.KVX_MATCH_KEEP_LAST])
def test_local_hits_far_past_the_published_span(flags):
    """Every block resident locally, the published spans cut early (flipped hashes) or absent
    (expired sessions): the local prefix runs far past the remote one, over many windows of 32, so the
    match has to continue the session's own chain there, from the first unmatched block."""
    w = kvx_inputs.bidir_mla_fp8(seed=29, n_sessions=32, n_layers=1, system_tokens=512, hist_range=(2000, 12000),
                                 resident_p=1.0, threshold=64)
    trim_to_blocks(w, set(range(0, w.n_sessions, 3)))
    c = Case(w, flip_frac=0.02, seed=11)
    expiry = np.where(np.arange(w.n_sessions) % 2 == 0, 50, 500).astype(np.int64)   # even sessions expired
    for exp in (None, expiry):
        want = c.oracle_match(flags=flags, expiry=exp, now=100)
        assert want["status"] == 0
        n_full = (np.diff(w.tok_off) // w.block_size)
        assert (want["local_hit"] == n_full).all()                           # all resident: to the end
        assert (want["remote_hit"] < n_full - 40).sum() >= 8                 # many spans end far earlier
        st, plan, got = c.match(want_plan=False, flags=flags, expiry=exp, now=100)
        assert st in (kvx.KVX_OK, kvx.KVX_ENOMEM) and plan is None
        assert_decisions(got, want)
    c.close()


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_match_decisions_at_block_sizes(bs):
    """Synthetic sessions at several block sizes (256 is past the shared-memory staging of the
    match): published hashes from the oracle with some flipped, a random half of the blocks resident."""
    rng = np.random.default_rng(bs)
    lens = rng.integers(0, 40 * bs, 48)
    lens[:4] = [0, bs - 1, bs, 3 * bs]                                       # empty, short, exact
    tokens = rng.integers(0, 151936, int(lens.sum())).astype(np.uint32)
    tok_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    orc = oracle.load()
    hs = [orc.block_hashes(tokens[tok_off[s]:tok_off[s + 1]], bs) for s in range(len(lens))]
    allh = np.concatenate(hs)
    remote = allh.copy()
    remote[rng.random(len(allh)) < 0.01] ^= np.uint64(1)
    rem_off = np.concatenate([[0], np.cumsum([len(h) for h in hs])]).astype(np.int64)
    remote_blk = np.arange(len(allh), dtype=np.int32)
    keys = np.unique(allh[rng.random(len(allh)) < 0.5])
    free = np.arange(len(allh), dtype=np.int32)
    want = orc.match(tokens, tok_off, bs, keys, remote, remote_blk, rem_off, 2 * bs, free)
    table = kvx.kvx_table_build(dev(keys, np.uint64), dev(np.arange(len(keys), dtype=np.int32), np.int32), len(keys))
    out = torch.zeros(len(lens) * 24, dtype=torch.uint8, device="cuda")
    st, plan = kvx.kvx_match_prefix(dev(tokens, np.uint32), dev(tok_off, np.int64), len(lens), bs, table,
                                    dev(remote, np.uint64), dev(remote_blk, np.int32), dev(rem_off, np.int64), 2 * bs,
                                    dev(free, np.int32), len(free), None, None, out, want_plan=False)
    assert st == kvx.KVX_OK and want["status"] == 0
    assert_decisions(results(out, len(lens)), want)
    assert want["push"].sum() > 0 and (want["remote_hit"] < np.diff(rem_off)).sum() > 0
    kvx.kvx_table_destroy(table)


def test_match_plan_and_push_reduced():
    w = kvx_inputs.bidir_mla_fp8(seed=22, n_sessions=16, n_layers=3, system_tokens=256, hist_range=(64, 2500),
                                 resident_p=0.5, threshold=128)
    c = Case(w, flip_frac=0.005, seed=4)
    want = c.oracle_match()
    src, _ = device_pool(w.decode, "fp8_bytes", seed=5)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    reqs = oracle_requests(c, want)
    # the device-built runs are the oracle's maximal runs of each pushing session's block pairs
    orc = oracle.load()
    wr = [orc.block_runs(r[1], r[2]) for r in reqs]
    rs, rd, rl = kvx.kvx_plan_runs(plan)
    assert rs.tolist() == (np.concatenate([x[0] for x in wr]) * 64).tolist()
    assert rd.tolist() == (np.concatenate([x[1] for x in wr]) * 64).tolist()
    assert rl.tolist() == (np.concatenate([x[2] for x in wr]) * 64).tolist()
    side = torch.cuda.Stream(priority=-1)
    for layer in range(w.decode.n_layers):
        kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")], reqs,
                 range(w.decode.n_layers))
    kvx.kvx_plan_destroy(plan)
    c.close()


def test_match_plan_pushed_as_multi_layer_launches():
    """A device-built pull plan pushed with kvx_push_layers in launches of two layers each (the last
    launch one layer) equals the oracle on every layer."""
    w = kvx_inputs.bidir_mla_fp8(seed=27, n_sessions=12, n_layers=5, system_tokens=256, hist_range=(64, 2000),
                                 resident_p=0.5, threshold=128)
    c = Case(w, flip_frac=0.005, seed=6)
    want = c.oracle_match()
    src, _ = device_pool(w.decode, "fp8_bytes", seed=8)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    kvx.kvx_plan_set_opts(plan, {"layers_per_launch": 2, "flags": kvx.KVX_PLAN_TIMING})
    n0 = kvx.kvx_launch_count()
    kvx.kvx_push_layers(plan, 0, 5, torch.cuda.Stream())
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    assert kvx.kvx_launch_count() - n0 == 3 and len(kvx.kvx_plan_push_times_ns(plan)[0]) == 3
    check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")],
                 oracle_requests(c, want), range(5))
    kvx.kvx_plan_destroy(plan)
    c.close()


PULL_LAYOUTS = {
    # name: (decode side, prefill side) as (shards, heads per shard, layout); 8 heads of 128 bf16 each
    "hnd_same": ((1, 8, 1), (1, 8, 1)),
    "nhd_to_hnd": ((1, 8, 0), (1, 8, 1)),
    "hnd_to_nhd": ((1, 8, 1), (1, 8, 0)),
    "hnd_tp1_to_hnd_tp2": ((1, 8, 1), (2, 4, 1)),
    "nhd_tp4_to_hnd_tp1": ((4, 2, 0), (1, 8, 1)),
}


@pytest.mark.parametrize("name", sorted(PULL_LAYOUTS))
def test_match_plan_between_pools_of_other_layouts(name):
    """The decode->prefill plan between K/V pools of different layouts or head partitions (8 heads of
    128 bf16): identical spans when both sides are head-major alike, otherwise per-(block, head) tiles
    built on the device; the consumer equals the oracle's push of the same pairs."""
    w = kvx_inputs.bidir_mla_fp8(seed=23, n_sessions=12, n_layers=2, system_tokens=256, hist_range=(64, 1500),
                                 resident_p=0.5, threshold=128)
    c = Case(w, flip_frac=0.005, seed=9)
    want = c.oracle_match()
    (ss, sh, sl), (ds, dh, dl) = PULL_LAYOUTS[name]
    kv = dict(n_planes=2, head_dim=128, elem_bytes=2)
    dec = w.decode.replace(n_shards=ss, heads_per_shard=sh, layout=sl, **kv)
    pre = w.prefill.replace(n_shards=ds, heads_per_shard=dh, layout=dl, **kv)
    src, _ = device_pool(dec, "bf16_normal", seed=12)
    dst, _ = device_pool(pre, "canary_bf16_normal")
    st, plan, got = c.match(kvx.Pool(dec, src), kvx.Pool(pre, dst))
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    assert (kvx.kvx_plan_get_info(plan)["strided"] == 0) == (name == "hnd_same")
    side = torch.cuda.Stream(priority=-1)
    for layer in range(dec.n_layers):
        kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    per = pre.n_planes * pre.n_shards
    check_layers(dec, src, pre, dst, lambda l: [canary_host(pre, "bf16_normal") for _ in range(per)],
                 oracle_requests(c, want), range(dec.n_layers))
    kvx.kvx_plan_destroy(plan)
    c.close()


def test_match_plan_refuses_shard_counts_that_do_not_divide():
    w = kvx_inputs.bidir_mla_fp8(seed=24, n_sessions=4, n_layers=1, system_tokens=128, hist_range=(64, 600),
                                 resident_p=0.5, threshold=64)
    c = Case(w)
    kv = dict(n_planes=2, head_dim=64, elem_bytes=2)
    dec = w.decode.replace(n_shards=3, heads_per_shard=2, **kv)
    pre = w.prefill.replace(n_shards=2, heads_per_shard=3, layout=kvx_inputs.LAYOUT_HND, **kv)
    src, _ = device_pool(dec, "bf16_normal", seed=1)
    dst, _ = device_pool(pre, "canary_bf16_normal")
    with pytest.raises(kvx.KvxError) as ei:
        c.match(kvx.Pool(dec, src), kvx.Pool(pre, dst))
    assert ei.value.status == kvx.KVX_EUNSUPPORTED
    c.close()


def test_match_full_sessions_two_layers():
    """All 256 sessions of the bidirectional workload (1024 shared + U[2k,32k] history tokens each);
    the pool has 2 of its 48 layers so the whole push is checked against the oracle."""
    w = kvx_inputs.bidir_mla_fp8(n_layers=2)
    c = Case(w)
    want = c.oracle_match()
    src, _ = device_pool(w.decode, "fp8_bytes", seed=w.seed)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    assert want["push"].sum() == w.n_sessions                   # every session has > 512 missing tokens
    side = torch.cuda.Stream(priority=-1)
    for layer in range(2):
        kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")],
                 oracle_requests(c, want), range(2))
    kvx.kvx_plan_destroy(plan)
    c.close()


@pytest.mark.parametrize("l_rem,want_push", [(511, 0), (512, 1), (513, 1)])
def test_threshold_edges(l_rem, want_push):
    bs, n = 1, 600
    rng = np.random.default_rng(l_rem)
    toks = rng.integers(0, kvx_inputs.VOCAB, n).astype(np.uint32)
    h = oracle.load().block_hashes(toks, bs)
    remote = h.copy()
    remote[l_rem] ^= np.uint64(9)
    table = kvx.kvx_table_build(None, None, 0)
    out = torch.zeros(24, dtype=torch.uint8, device="cuda")
    st, plan = kvx.kvx_match_prefix(dev(toks, np.uint32), dev(np.array([0, n], np.int64), np.int64), 1, bs, table,
                                    dev(remote, np.uint64), dev(np.arange(n, dtype=np.int32), np.int32),
                                    dev(np.array([0, n], np.int64), np.int64), 512,
                                    dev(np.arange(n, dtype=np.int32), np.int32), n, None, None, out, want_plan=False)
    r = results(out, 1)[0]
    assert (r["local_hit_blocks"], r["remote_hit_blocks"], r["missing_tokens"], r["push"]) == (0, l_rem, l_rem, want_push)
    kvx.kvx_table_destroy(table)


def test_match_plan_with_nothing_to_push():
    """No session reaches the threshold, and a call with no sessions at all: each still returns a
    plan, with no runs; pushing it is a no-op that syncs DONE and leaves the prefill pool as it was."""
    w = kvx_inputs.bidir_mla_fp8(seed=26, n_sessions=6, n_layers=2, system_tokens=128, hist_range=(64, 900),
                                 resident_p=0.5, threshold=1 << 30)
    c = Case(w)
    want = c.oracle_match()
    assert want["push"].sum() == 0
    src, _ = device_pool(w.decode, "fp8_bytes", seed=2)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    before = [b.clone() for b in dst]
    for n_sessions in (w.n_sessions, 0):
        w.n_sessions = n_sessions
        st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
        assert st == kvx.KVX_OK and plan is not None
        if n_sessions:
            assert_decisions(got, want)
        assert kvx.kvx_plan_get_info(plan)["n_runs"] == 0
        for layer in range(2):
            kvx.kvx_push_layer(plan, layer, torch.cuda.current_stream())
        assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
        assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE] * 2
        kvx.kvx_plan_destroy(plan)
    assert all(torch.equal(a, b) for a, b in zip(before, dst))
    c.close()


@pytest.mark.parametrize("entry", ["decisions", "plan", "static"])
@pytest.mark.parametrize("bad", ["token_range_past_total", "negative_remote_total", "remote_ranges_overlap"])
def test_match_rejects_malformed_offsets(entry, bad):
    """CSR offsets that do not describe the arrays are refused with KVX_EINVAL: the kernels bound every
    read by the CSR totals (read on the device), flag the session and read nothing out of range."""
    bs, n = 4, 3
    toks = np.arange(48, dtype=np.uint32)
    tok_off = np.array([0, 16, 32, 48], np.int64)
    rem_off = np.array([0, 4, 8, 12], np.int64)
    if bad == "token_range_past_total":
        tok_off = np.array([0, 16, 60, 48], np.int64)
    elif bad == "negative_remote_total":
        rem_off = np.array([0, 4, 8, -1], np.int64)
    else:
        rem_off = np.array([0, 8, 4, 12], np.int64)
    remote = np.zeros(12, np.uint64)
    table = kvx.kvx_table_build(None, None, 0)
    out = torch.zeros(n * 24, dtype=torch.uint8, device="cuda")
    args = (dev(toks, np.uint32), dev(tok_off, np.int64), n, bs, table, dev(remote, np.uint64))
    with pytest.raises(kvx.KvxError) as ei:
        if entry == "static":
            kvx.kvx_match_prefix_static(*args, dev(rem_off, np.int64), 4, 100, out)
        else:
            g = PoolGeom(1, 1, 1, 1, 16, 1, bs, 64)
            pools = [kvx.Pool(g, [torch.zeros(g.buffer_bytes, dtype=torch.uint8, device="cuda")]) for _ in range(2)]
            kvx.kvx_match_prefix(*args, dev(np.arange(12, dtype=np.int32), np.int32), dev(rem_off, np.int64), 4,
                                 dev(np.arange(64, dtype=np.int32), np.int32), 64, pools[0], pools[1], out,
                                 want_plan=entry == "plan")
    assert ei.value.status == kvx.KVX_EINVAL
    kvx.kvx_table_destroy(table)


def test_free_list_too_short_is_enomem():
    w = kvx_inputs.bidir_mla_fp8(seed=23, n_sessions=8, n_layers=1, system_tokens=128, hist_range=(600, 1500),
                                 resident_p=0.3, threshold=64)
    c = Case(w)
    full = c.oracle_match()
    need = int(sum(full["missing"][full["push"] == 1]) // 64)
    short = c.oracle_match(n_free=need - 1)
    assert short["status"] == 5
    src, _ = device_pool(w.decode, "fp8_bytes", seed=1)
    dst, big = device_pool(w.prefill, "canary_fp8_bytes")
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst), n_free=need - 1)
    assert st == kvx.KVX_ENOMEM and plan is None
    assert_decisions(got, short)
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst), n_free=need)
    assert st == kvx.KVX_OK and plan is not None
    kvx.kvx_plan_destroy(plan)
    c.close()


def test_bad_free_block_fails_the_layer_without_writing_outside():
    """A free-list entry outside the prefill pool: the copy kernel's bounds guard skips those tiles and
    kvx_sync reports the layer FAILED; nothing outside the pool buffers changes."""
    w = kvx_inputs.bidir_mla_fp8(seed=24, n_sessions=2, n_layers=1, system_tokens=128, hist_range=(600, 900),
                                 resident_p=0.0, threshold=64)
    bad_free = w.free_blocks.copy()
    bad_free[0] = w.prefill.n_blocks + 5
    w.free_blocks = bad_free
    c = Case(w)
    src, _ = device_pool(w.decode, "fp8_bytes", seed=1)
    per = -(-w.prefill.buffer_bytes // 512) * 512
    guard = torch.full((per * 3,), 0x55, dtype=torch.uint8, device="cuda")
    dst = [guard[per:per + w.prefill.buffer_bytes]]
    dst[0].fill_(kvx_inputs.CANARY_FP8)
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
    assert st == kvx.KVX_OK
    kvx.kvx_push_layer(plan, 0, torch.cuda.current_stream())
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_EFAILED
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_FAILED]
    assert bool((guard[:per] == 0x55).all()) and bool((guard[per + w.prefill.buffer_bytes:] == 0x55).all())
    kvx.kvx_plan_destroy(plan)
    c.close()


def test_bidir_full_scale_in_waves():
    """The full bidirectional workload: 256 sessions, 48 layers of fp8 576-byte latents (decode pool
    ~130 GB, prefill pool ~85 GB). Sessions are matched and pushed in 4 waves of 64 into one recycled
    free region; after each wave, layers 0, 23 and 47 are checked whole against the oracle."""
    orc = oracle.load()
    w0 = kvx_inputs.bidir_mla_fp8(n_layers=48, free_blocks=1)        # sizes only
    hs = [orc.block_hashes(w0.tokens[w0.tok_off[s]:w0.tok_off[s + 1]], 64) for s in range(w0.n_sessions)]
    allh = np.concatenate(hs)
    keys = np.unique(allh[w0.resident])
    waves = [range(i, i + 64) for i in range(0, 256, 64)]
    # free region large enough for the largest wave (decisions from the oracle)
    need = []
    for wv in waves:
        s0, s1 = wv[0], wv[-1] + 1
        sub = orc.match(w0.tokens[w0.tok_off[s0]:w0.tok_off[s1]], w0.tok_off[s0:s1 + 1] - w0.tok_off[s0], 64, keys,
                        allh[w0.rem_off[s0]:w0.rem_off[s1]], w0.remote_blk[w0.rem_off[s0]:w0.rem_off[s1]],
                        w0.rem_off[s0:s1 + 1] - w0.rem_off[s0], w0.threshold, np.zeros(0, np.int32))
        need.append(int(sub["missing"][sub["push"] == 1].sum() // 64))
    w = kvx_inputs.bidir_mla_fp8(n_layers=48, free_blocks=max(need))
    assert np.array_equal(w.tokens, w0.tokens) and np.array_equal(w.remote_blk, w0.remote_blk)
    src, _ = device_pool(w.decode, "fp8_bytes", seed=w.seed)
    dst, dbig = device_pool(w.prefill, "canary_fp8_bytes")
    table = kvx.kvx_table_build(dev(keys, np.uint64), dev(np.arange(len(keys), dtype=np.int32), np.int32), len(keys))
    sp, dp = kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst)
    side = torch.cuda.Stream()
    for wv in waves:
        s0, s1 = wv[0], wv[-1] + 1
        t0, t1, r0, r1 = w.tok_off[s0], w.tok_off[s1], w.rem_off[s0], w.rem_off[s1]
        toks, tok_off = w.tokens[t0:t1], w.tok_off[s0:s1 + 1] - t0
        rh, rb, rem_off = allh[r0:r1], w.remote_blk[r0:r1], w.rem_off[s0:s1 + 1] - r0
        want = orc.match(toks, tok_off, 64, keys, rh, rb, rem_off, w.threshold, w.free_blocks)
        assert want["status"] == 0
        kvx_inputs.fill_canary(dbig, "fp8_bytes")                       # recycle the free region
        out = torch.zeros(64 * 24, dtype=torch.uint8, device="cuda")
        st, plan = kvx.kvx_match_prefix(dev(toks, np.uint32), dev(tok_off, np.int64), 64, 64, table,
                                        dev(rh, np.uint64), dev(rb, np.int32), dev(rem_off, np.int64), w.threshold,
                                        dev(w.free_blocks, np.int32), len(w.free_blocks), sp, dp, out)
        assert st == kvx.KVX_OK
        assert_decisions(results(out, 64), want)
        for layer in range(48):
            kvx.kvx_push_layer(plan, layer, side)
        assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
        reqs, k = [], 0
        for s in range(64):
            if want["push"][s]:
                nb = int(want["missing"][s]) // 64
                reqs.append((nb * 64, want["pair_src"][k:k + nb], want["pair_dst"][k:k + nb]))
                k += nb
        check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")], reqs, [0, 23, 47])
        kvx.kvx_plan_destroy(plan)
    kvx.kvx_table_destroy(table)



@pytest.mark.parametrize("flags,ttl", [(kvx.KVX_MATCH_FILL_HOLES, False), (kvx.KVX_MATCH_KEEP_LAST, False),
                                       (0, True), (kvx.KVX_MATCH_FILL_HOLES | kvx.KVX_MATCH_KEEP_LAST, True)],
                         ids=["holes", "keep_last", "ttl", "all"])
def test_match_options_plan_and_push(flags, ttl):
    w = kvx_inputs.bidir_mla_fp8(seed=25, n_sessions=20, n_layers=2, system_tokens=256, hist_range=(0, 2500),
                                 resident_p=0.5, threshold=128)
    trim_to_blocks(w, [0, 3, 7, 12])          # these end on a block boundary, so keep-last applies
    c = Case(w, flip_frac=0.003, seed=6)
    expiry = np.random.default_rng(8).integers(0, 200, w.n_sessions) if ttl else None
    want = c.oracle_match(flags=flags, expiry=expiry, now=100)
    assert want["status"] == 0 and want["push"].sum() > 2
    src, _ = device_pool(w.decode, "fp8_bytes", seed=5)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst), flags=flags, expiry=expiry, now=100)
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    orc = oracle.load()
    reqs = oracle_requests(c, want)
    wr = [orc.block_runs(r[1], r[2]) for r in reqs]
    rs, rd, rl = kvx.kvx_plan_runs(plan)
    assert rs.tolist() == (np.concatenate([x[0] for x in wr]) * 64).tolist()
    assert rd.tolist() == (np.concatenate([x[1] for x in wr]) * 64).tolist()
    assert rl.tolist() == (np.concatenate([x[2] for x in wr]) * 64).tolist()
    side = torch.cuda.Stream()
    for layer in range(2):
        kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")], reqs, range(2))
    kvx.kvx_plan_destroy(plan)
    c.close()


def test_plan_scan_wait_runs_out_then_next_call_is_exact():
    """KVX_MATCH_TEST_SCAN_STALL: the first tile of the look-back scan that numbers the plan's runs
    publishes nothing, so the next tile's bounded wait (1 ms under the hook) runs out; the call returns
    KVX_ETIMEDOUT with no plan and nothing faults. The same call without the hook then gives the
    oracle's decisions and a plan whose pushed bytes equal the oracle's."""
    w = kvx_inputs.bidir_mla_fp8(seed=26, n_sessions=24, n_layers=1, system_tokens=256, hist_range=(2000, 6000),
                                 resident_p=0.3, threshold=64)
    assert w.rem_off[-1] > 1024                                  # the run scan has more than one tile
    c = Case(w)
    src, _ = device_pool(w.decode, "fp8_bytes", seed=5)
    dst, _ = device_pool(w.prefill, "canary_fp8_bytes")
    with pytest.raises(kvx.KvxError) as ei:
        c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst), flags=kvx.KVX_MATCH_TEST_SCAN_STALL)
    assert ei.value.status == kvx.KVX_ETIMEDOUT
    want = c.oracle_match()
    assert want["status"] == 0 and want["push"].sum() > 1
    st, plan, got = c.match(kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst))
    assert st == kvx.KVX_OK
    assert_decisions(got, want)
    kvx.kvx_push_layer(plan, 0, torch.cuda.Stream())
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.decode, src, w.prefill, dst, lambda l: [canary_host(w.prefill, "fp8_bytes")],
                 oracle_requests(c, want), range(1))
    kvx.kvx_plan_destroy(plan)
    c.close()
