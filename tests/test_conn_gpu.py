"""Chunked prefill through the connector and the device push, checked byte for byte against the
oracle.

A request's prefill runs in chunks; each chunk's forward pass (the fixture kernel, one launch per
layer and plane) rewrites that chunk's producer blocks after a long dependent spin. Following the
"vLLM MoRIIO KV Connector" notes, section 3.2 (chunked prefill collects blocks until the last chunk
before writing; a write task without destination ids waits on the deferred list), the connector
keeps the request out of READY until the last chunk, so no push is issued earlier; the pushes of
the last chunk's forward are gated per layer on that layer's event and cover the blocks of every
chunk. Per-layer states feed the connector's write reports (section 6, batch state), and an
injected failure turns into load errors for the consumer to recompute (section 3.1)."""
import numpy as np
import pytest

import kvx_inputs
import prefill_fixture
from gpu_helpers import canary_host, check_layers, device_pool, layer_buffers

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
kvx = pytest.importorskip("disaggregated_prefill_decode_gb300.kvx")


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


SRC = kvx_inputs.PoolGeom(n_layers=4, n_planes=2, n_shards=1, heads_per_shard=8, head_dim=128, elem_bytes=2,
                          block_size=16, n_blocks=64)
CHUNKS = [np.arange(4, 8), np.arange(12, 16), np.arange(20, 23)]      # producer blocks per chunk
N_TOKENS = [64, 128, 168]                                             # computed length after each chunk


def forward_chunk(src_bufs, c, main, spin):
    """The chunk's forward pass: per layer, rewrite the chunk's blocks in both planes; one event per
    layer recorded after it."""
    ids = CHUNKS[c]
    bb = SRC.block_size * SRC.row_bytes
    lo, hi = int(ids[0]) * bb, (int(ids[-1]) + 1) * bb
    events = []
    for layer in range(SRC.n_layers):
        for p, b in enumerate(layer_buffers(SRC, src_bufs, layer)):
            prefill_fixture.prefill(16, spin, b[lo:hi], hi - lo, seed=1000 * c + 10 * layer + p, stream=main)
        ev = torch.cuda.Event()
        ev.record(main)
        events.append(ev)
    return events


def dst_geom(bs):
    return SRC.replace(block_size=bs, n_blocks=64 * 16 // bs)


def dst_ids_for(bs):
    n = -(-N_TOKENS[-1] // bs)
    return np.random.default_rng(bs).permutation(dst_geom(bs).n_blocks)[:n].astype(np.int32)


def run_chunked(bs, register_first, inject_layer=None, spin=20000):
    dgeom = dst_geom(bs)
    src, _ = device_pool(SRC, "bf16_normal", seed=77)
    dst, _ = device_pool(dgeom, "canary_bf16_normal")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=-1)
    conn = kvx.kvx_conn_create()
    rid, now = 42, 0
    dst_ids = dst_ids_for(bs)
    if register_first:
        kvx.kvx_conn_register(conn, rid, 0, dst_ids, now)
    plan, writes = None, []
    launches_before, fixtures_before = kvx.kvx_launch_count(), prefill_fixture.launch_count()
    for c in range(len(CHUNKS)):
        last = c == len(CHUNKS) - 1
        kvx.kvx_conn_prefill(conn, rid, 0, CHUNKS[c], N_TOKENS[c], last, now)
        events = forward_chunk(src, c, main, spin)
        if not last:
            # the gate: nothing may move before the last chunk
            assert kvx.kvx_conn_get(conn, rid)["state"] == kvx.KVX_CONN_WAITING
            assert kvx.kvx_conn_poll(conn, now) == []
            assert kvx.kvx_launch_count() == launches_before                  # no push launched yet
            continue
        if kvx.kvx_conn_get(conn, rid)["state"] == kvx.KVX_CONN_READY:
            # layer-wise: the pushes of the last chunk's forward, one per layer, gated on its event
            plan = start_plan(conn, rid, src, dst, dgeom, inject_layer, now)
            for layer in range(SRC.n_layers):
                kvx.kvx_push_layer(plan, layer, side, events[layer])
                kvx.kvx_conn_write_issued(conn, rid, 0, 0, 1)
                writes.append((layer, layer + 1))
        else:
            assert kvx.kvx_conn_get(conn, rid)["state"] == kvx.KVX_CONN_DEFERRED
            deferred_after = events[-1]
    # one forward launch per (chunk, layer, plane), counted by the fixture's own library
    assert prefill_fixture.launch_count() - fixtures_before == len(CHUNKS) * SRC.n_layers * SRC.n_planes
    if not register_first:
        # the deferred task: the registration arrives after the forward; all layers in one write,
        # gated on the event after the last layer (one stream: it follows every layer)
        now += 1000
        kvx.kvx_conn_register(conn, rid, 0, dst_ids, now)
        assert kvx.kvx_conn_poll(conn, now) == [(rid, 0, kvx.KVX_CONN_READY)]
        plan = start_plan(conn, rid, src, dst, dgeom, inject_layer, now)
        kvx.kvx_push_layers(plan, 0, SRC.n_layers, side, deferred_after)
        kvx.kvx_conn_write_issued(conn, rid, 0, 0, 1)
        writes.append((0, SRC.n_layers))
    kvx.kvx_conn_seal(conn, rid, 0, 0)
    st = kvx.kvx_sync(plan, -1)
    states = kvx.kvx_plan_layer_states(plan)
    for l0, l1 in writes:
        kvx.kvx_conn_write_done(conn, rid, 0, 0, states[l0:l1], now_us=now)
    return conn, rid, plan, st, src, dst, dgeom, dst_ids


def start_plan(conn, rid, src, dst, dgeom, inject_layer, now):
    kvx.kvx_conn_start(conn, rid, 0, now)
    src_ids, dst_ids = kvx.kvx_conn_ids(conn, rid)
    assert np.array_equal(src_ids, np.concatenate(CHUNKS))            # blocks of every chunk
    n_tok = kvx.kvx_conn_get(conn, rid)["n_tokens"]
    plan = kvx.kvx_plan(kvx.Pool(SRC, src), kvx.Pool(dgeom, dst), [(n_tok, src_ids, dst_ids)])
    if inject_layer is not None:
        kvx.kvx_plan_inject_failure(plan, inject_layer)
    return plan


@pytest.mark.parametrize("register_first", [True, False], ids=["registered_first", "deferred"])
@pytest.mark.parametrize("bs", [16, 64])
def test_chunked_prefill_push_through_the_connector(bs, register_first):
    conn, rid, plan, st, src, dst, dgeom, dst_ids = run_chunked(bs, register_first)
    assert st == kvx.KVX_OK
    events = kvx.kvx_conn_poll(conn, 10**9)
    assert events[-1] == (rid, 0, kvx.KVX_CONN_DONE)
    info = kvx.kvx_conn_get(conn, rid)
    assert info["writes_done"] == info["writes_expected"] == (SRC.n_layers if register_first else 1)
    check_layers(SRC, src, dgeom, dst, lambda l: [canary_host(dgeom, "bf16_normal") for _ in range(2)],
                 [(N_TOKENS[-1], np.concatenate(CHUNKS), dst_ids)], range(SRC.n_layers))
    kvx.kvx_plan_destroy(plan)
    kvx.kvx_conn_release(conn, rid)
    kvx.kvx_conn_destroy(conn)


@pytest.mark.parametrize("register_first", [True, False], ids=["registered_first", "deferred"])
def test_failed_layer_becomes_load_errors(register_first):
    conn, rid, plan, st, src, dst, dgeom, dst_ids = run_chunked(16, register_first, inject_layer=2, spin=2000)
    assert st == kvx.KVX_EFAILED
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE] * 2 + [kvx.KVX_LAYER_FAILED] + \
        [kvx.KVX_LAYER_DONE]
    assert kvx.kvx_conn_poll(conn, 10**9)[-1] == (rid, 0, kvx.KVX_CONN_FAILED)
    info = kvx.kvx_conn_get(conn, rid)
    assert info["writes_failed"] == 1 and info["first_error"] == 0
    assert np.array_equal(kvx.kvx_conn_load_errors(conn, rid), dst_ids)   # every block of the request
    kvx.kvx_plan_destroy(plan)
    kvx.kvx_conn_destroy(conn)
