"""kvx_match_prefix_static: the match decision for callers that cannot allocate device memory on the
request path (serving engines that hand nearly all free HBM to their KV pools at start-up, where a
later allocation can fail and cudaMalloc / cudaFree can stall the other streams).

Through the C-ABI, the allocation-free entry point must give exactly the decisions of the oracle
(integers: bit-exact, field by field) and of kvx_match_prefix, on two calls in a row, since both
calls share one fixed scratch array that keeps the previous call's contents. The two entry points
launch the same match kernel, so the oracle is the checker that a fault they share cannot pass.
This file sorts last so that a run stopping at its first failure has already run every other test;
it also passes alone in a fresh process."""
import numpy as np
import pytest

import kvx_inputs
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
kvx = pytest.importorskip("disaggregated_prefill_decode_gb300.kvx")


def dev(a):
    a = np.ascontiguousarray(a)
    view = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
    if len(a) == 0:
        a = np.zeros(1, a.dtype)
    return torch.from_numpy(a.view(view)).to("cuda")


def workload(seed, n_sessions, threshold):
    w = kvx_inputs.bidir_mla_fp8(seed=seed, n_sessions=n_sessions, n_layers=1, system_tokens=256,
                                 hist_range=(64, 4000), resident_p=0.6, threshold=threshold)
    orc = oracle.load()
    hs = np.concatenate([orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], 64) for s in range(w.n_sessions)])
    remote = hs.copy()
    flip = np.random.default_rng(seed).random(len(hs)) < 0.01       # some published hashes disagree
    remote[flip] ^= np.uint64(1)
    keys = np.unique(hs[w.resident])
    table = kvx.kvx_table_build(dev(keys), dev(np.arange(len(keys), dtype=np.int32)), len(keys))
    return w, remote, table, keys


def oracle_decisions(w, remote, keys, n_free):
    """The oracle's decisions, with a free list of n_free blocks (the first n_free of the workload's)."""
    return oracle.load().match(w.tokens, w.tok_off, 64, keys, remote, w.remote_blk, w.rem_off, w.threshold,
                               w.free_blocks[:n_free])


def assert_matches_oracle(got, want):
    res = got.view(kvx.MATCH_RESULT_DTYPE)
    for field, key in (("local_hit_blocks", "local_hit"), ("remote_hit_blocks", "remote_hit"),
                       ("missing_tokens", "missing"), ("push", "push"), ("dst_start", "dst_start")):
        assert res[field].tolist() == want[key].tolist(), field


def decisions_with_allocation(w, remote, table, n_free):
    out = torch.zeros(w.n_sessions * 24, dtype=torch.uint8, device="cuda")
    st, plan = kvx.kvx_match_prefix(dev(w.tokens), dev(w.tok_off), w.n_sessions, 64, table, dev(remote),
                                    dev(w.remote_blk), dev(w.rem_off), w.threshold, dev(w.free_blocks), n_free,
                                    None, None, out, want_plan=False)
    return st, out.cpu().numpy()


def decisions_without_allocation(w, remote, table, n_free):
    out = torch.full((w.n_sessions * 24,), 0x5A, dtype=torch.uint8, device="cuda")   # no stale zeros to hide behind
    st = kvx.kvx_match_prefix_static(dev(w.tokens), dev(w.tok_off), w.n_sessions, 64, table, dev(remote),
                                     dev(w.rem_off), w.threshold, n_free, out)
    return st, out.cpu().numpy()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_static_scratch_matches_allocating_entry_point_twice():
    cases = [workload(31, 40, 256), workload(32, 300, 64)]     # second call: different size, same array
    for w, remote, table, keys in cases:
        n_free = len(w.free_blocks)
        ref = oracle_decisions(w, remote, keys, n_free)
        assert ref["status"] == 0
        st_a, want = decisions_with_allocation(w, remote, table, n_free)
        st_b, got = decisions_without_allocation(w, remote, table, n_free)
        assert st_a == st_b == kvx.KVX_OK
        assert_matches_oracle(got, ref)
        assert np.array_equal(got, want)
        res = got.view(kvx.MATCH_RESULT_DTYPE)
        assert res["push"].sum() > 0 and (res["push"] == 0).sum() > 0
    # a free list too short for the pushes: KVX_ENOMEM from both, and the oracle's decisions for that
    # free list (its status 5: too short; the decisions and dst_start positions are still written)
    w, remote, table, keys = cases[1]
    ref = oracle_decisions(w, remote, keys, 5)
    assert ref["status"] == 5
    st_a, want = decisions_with_allocation(w, remote, table, 5)
    st_b, got = decisions_without_allocation(w, remote, table, 5)
    assert st_a == st_b == kvx.KVX_ENOMEM
    assert_matches_oracle(got, ref)
    assert np.array_equal(got, want)
    for _, _, table, _ in cases:
        kvx.kvx_table_destroy(table)


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_static_scratch_rejects_too_many_sessions():
    table = kvx.kvx_table_build(None, None, 0)
    tiny = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(kvx.KvxError) as ei:
        kvx.kvx_match_prefix_static(tiny, tiny, 65537, 64, table, tiny, tiny, 512, 0, tiny)
    assert ei.value.status == kvx.KVX_EINVAL and "65536" in str(ei.value)
    kvx.kvx_table_destroy(table)
