"""Connector state machine (kvx_conn_*), host only, driven by a fake microsecond clock.

The protocol is the one of the push-mode NIXL connector article, "Implementierungsdetails" steps
1-3 (registration at allocation; rendezvous in either order by request id, coping with resent,
preempted and retried requests; one completion per producer rank), and of the "vLLM MoRIIO KV
Connector" notes, sections 3.1 (failed loads are recomputed), 3.2 (deferred tasks given up after
defer_timeout; chunked prefill collects blocks until the last chunk; the write count is sealed at
the number actually queued), 5 (timeout defaults 30 s / 60 s / 120 s) and 6 (batch state over all
layers; consumer_tp / producer_tp acknowledgements)."""
import random
import threading
import time

import numpy as np
import pytest

kvx = pytest.importorskip("disaggregated_prefill_decode_gb300.kvx")

S = 1_000_000   # one second on the fake clock
DONE, FAILED, PENDING, IDLE = kvx.KVX_LAYER_DONE, kvx.KVX_LAYER_FAILED, kvx.KVX_LAYER_PENDING, kvx.KVX_LAYER_IDLE


@pytest.fixture
def conn():
    c = kvx.kvx_conn_create()
    yield c
    kvx.kvx_conn_destroy(c)


def state(c, rid):
    return kvx.kvx_conn_get(c, rid)["state"]


def status_of(fn, *args, **kw):
    try:
        fn(*args, **kw)
        return kvx.KVX_OK
    except kvx.KvxError as e:
        return e.status


def finish(c, rid, attempt, n_writes=1, states=(DONE,), now=0, rank=0):
    kvx.kvx_conn_start(c, rid, attempt, now)
    kvx.kvx_conn_write_issued(c, rid, attempt, rank, n_writes)
    kvx.kvx_conn_seal(c, rid, attempt, rank)
    for _ in range(n_writes):
        kvx.kvx_conn_write_done(c, rid, attempt, rank, list(states), now_us=now)


def test_registration_first_then_prefill(conn):
    kvx.kvx_conn_register(conn, 7, 0, [40, 41, 42], now_us=0)
    assert state(conn, 7) == kvx.KVX_CONN_WAITING              # held until the producer's prefill ends
    assert kvx.kvx_conn_poll(conn, 1 * S) == []
    kvx.kvx_conn_prefill(conn, 7, 0, [3, 4, 5], n_tokens=40, last_chunk=True, now_us=2 * S)
    assert kvx.kvx_conn_poll(conn, 2 * S) == [(7, 0, kvx.KVX_CONN_READY)]
    src, dst = kvx.kvx_conn_ids(conn, 7)
    assert list(src) == [3, 4, 5] and list(dst) == [40, 41, 42]
    assert kvx.kvx_conn_get(conn, 7)["n_tokens"] == 40


def test_prefill_first_then_registration(conn):
    kvx.kvx_conn_prefill(conn, 8, 0, [9, 10], n_tokens=20, last_chunk=True, now_us=0)
    assert state(conn, 8) == kvx.KVX_CONN_DEFERRED             # producer holds its blocks
    assert kvx.kvx_conn_poll(conn, 59 * S) == []
    kvx.kvx_conn_register(conn, 8, 0, [1, 2], now_us=59 * S)
    assert kvx.kvx_conn_poll(conn, 59 * S) == [(8, 0, kvx.KVX_CONN_READY)]
    assert kvx.kvx_conn_poll(conn, 178 * S) == []             # the defer deadline no longer applies
    assert kvx.kvx_conn_poll(conn, 179 * S) == [(8, 0, kvx.KVX_CONN_ABORTED)]   # never started: abort


def test_defer_timeout_expires_exactly_at_the_deadline(conn):
    kvx.kvx_conn_prefill(conn, 1, 0, [5], n_tokens=3, last_chunk=True, now_us=10)
    assert kvx.kvx_conn_poll(conn, 10 + 60 * S - 1) == []      # default defer_timeout: 60 s
    assert kvx.kvx_conn_poll(conn, 10 + 60 * S) == [(1, 0, kvx.KVX_CONN_EXPIRED)]
    # a registration after the producer gave up is told so; the record stays EXPIRED
    assert status_of(kvx.kvx_conn_register, conn, 1, 0, [9], 61 * S) == kvx.KVX_ETIMEDOUT
    assert state(conn, 1) == kvx.KVX_CONN_EXPIRED
    assert kvx.kvx_conn_poll(conn, 1000 * S) == []


def test_custom_timeouts():
    c = kvx.kvx_conn_create(defer_timeout_us=5, transfer_timeout_us=7, recv_abort_timeout_us=11)
    kvx.kvx_conn_prefill(c, 1, 0, [0], 1, True, now_us=0)
    kvx.kvx_conn_register(c, 2, 0, [0], now_us=0)
    kvx.kvx_conn_prefill(c, 3, 0, [0], 1, True, now_us=0)
    kvx.kvx_conn_register(c, 3, 0, [0], now_us=0)
    kvx.kvx_conn_start(c, 3, 0, now_us=1)
    assert kvx.kvx_conn_poll(c, 4) == [(3, 0, kvx.KVX_CONN_READY)]
    assert kvx.kvx_conn_poll(c, 5) == [(1, 0, kvx.KVX_CONN_EXPIRED)]
    assert kvx.kvx_conn_poll(c, 8) == [(3, 0, kvx.KVX_CONN_TIMED_OUT)]
    assert kvx.kvx_conn_poll(c, 11) == [(2, 0, kvx.KVX_CONN_ABORTED)]
    kvx.kvx_conn_destroy(c)


def test_transfer_and_abort_default_timeouts(conn):
    kvx.kvx_conn_register(conn, 1, 0, [0], now_us=0)           # prefill never finishes
    kvx.kvx_conn_register(conn, 2, 0, [1], now_us=0)
    kvx.kvx_conn_prefill(conn, 2, 0, [1], 16, True, now_us=0)
    kvx.kvx_conn_start(conn, 2, 0, now_us=1 * S)
    assert kvx.kvx_conn_poll(conn, 31 * S - 1) == [(2, 0, kvx.KVX_CONN_READY)]
    assert kvx.kvx_conn_poll(conn, 31 * S) == [(2, 0, kvx.KVX_CONN_TIMED_OUT)]     # transfer_timeout 30 s
    assert kvx.kvx_conn_poll(conn, 120 * S - 1) == []
    assert kvx.kvx_conn_poll(conn, 120 * S) == [(1, 0, kvx.KVX_CONN_ABORTED)]      # recv_abort_timeout 120 s
    # late reports of a timed-out transfer are refused, not counted
    assert status_of(kvx.kvx_conn_write_issued, conn, 2, 0, 0, 1) == kvx.KVX_EINVAL


def test_abort_does_not_fire_after_completion(conn):
    kvx.kvx_conn_register(conn, 4, 0, [1], now_us=0)
    kvx.kvx_conn_prefill(conn, 4, 0, [2], 16, True, now_us=0)
    finish(conn, 4, 0, now=1)
    assert kvx.kvx_conn_poll(conn, 10_000 * S) == [(4, 0, kvx.KVX_CONN_READY), (4, 0, kvx.KVX_CONN_DONE)]


def test_resent_registration_is_idempotent(conn):
    kvx.kvx_conn_register(conn, 3, 0, [1, 2, 3], now_us=0)
    kvx.kvx_conn_register(conn, 3, 0, [1, 2, 3], now_us=5)
    assert status_of(kvx.kvx_conn_register, conn, 3, 0, [1, 2, 4], 6) == kvx.KVX_EINVAL
    kvx.kvx_conn_prefill(conn, 3, 0, [8], 16, True, now_us=7)
    kvx.kvx_conn_register(conn, 3, 0, [1, 2, 3], now_us=8)     # resent after READY: still one event
    assert kvx.kvx_conn_poll(conn, 9) == [(3, 0, kvx.KVX_CONN_READY)]


def test_retried_request_starts_over_and_ignores_the_old_attempt(conn):
    kvx.kvx_conn_register(conn, 5, 0, [10, 11], now_us=0)
    kvx.kvx_conn_prefill(conn, 5, 0, [1, 2], 32, True, now_us=0)
    kvx.kvx_conn_start(conn, 5, 0, now_us=1)
    kvx.kvx_conn_write_issued(conn, 5, 0, 0, 2)
    # the consumer preempted the request and registers it again with new blocks
    kvx.kvx_conn_register(conn, 5, 1, [20, 21], now_us=2)
    info = kvx.kvx_conn_get(conn, 5)
    assert (info["attempt"], info["state"], info["writes_issued"]) == (1, kvx.KVX_CONN_WAITING, 0)
    # stale reports and chunks of attempt 0 change nothing
    kvx.kvx_conn_write_done(conn, 5, 0, 0, [DONE], now_us=3)
    kvx.kvx_conn_seal(conn, 5, 0, 0)
    kvx.kvx_conn_prefill(conn, 5, 0, [99], 48, True, now_us=3)
    kvx.kvx_conn_register(conn, 5, 0, [77], now_us=3)
    assert kvx.kvx_conn_get(conn, 5)["state"] == kvx.KVX_CONN_WAITING
    # the READY event of attempt 0 was never polled: it is dropped with the old attempt
    assert kvx.kvx_conn_poll(conn, 4) == []
    kvx.kvx_conn_prefill(conn, 5, 1, [3, 4], 32, True, now_us=5)
    assert kvx.kvx_conn_poll(conn, 5) == [(5, 1, kvx.KVX_CONN_READY)]
    src, dst = kvx.kvx_conn_ids(conn, 5)
    assert list(src) == [3, 4] and list(dst) == [20, 21]
    # the first attempt's transfer deadline does not fire on the second attempt
    kvx.kvx_conn_start(conn, 5, 1, now_us=100 * S)
    assert kvx.kvx_conn_poll(conn, 31 * S + 10) == []


def test_newer_attempt_from_the_producer_side(conn):
    kvx.kvx_conn_prefill(conn, 6, 0, [1], 16, True, now_us=0)      # DEFERRED
    kvx.kvx_conn_prefill(conn, 6, 1, [2], 16, False, now_us=1)     # retried prefill, first chunk
    assert state(conn, 6) == kvx.KVX_CONN_WAITING
    assert kvx.kvx_conn_poll(conn, 61 * S) == []                   # the old defer deadline is void


def test_chunked_prefill_moves_nothing_before_the_last_chunk(conn):
    kvx.kvx_conn_register(conn, 9, 0, [30, 31, 32, 33], now_us=0)
    kvx.kvx_conn_prefill(conn, 9, 0, [0, 1], n_tokens=32, last_chunk=False, now_us=1)
    kvx.kvx_conn_prefill(conn, 9, 0, [2], n_tokens=48, last_chunk=False, now_us=2)
    assert state(conn, 9) == kvx.KVX_CONN_WAITING and kvx.kvx_conn_poll(conn, 3) == []
    assert status_of(kvx.kvx_conn_start, conn, 9, 0, 3) == kvx.KVX_EINVAL
    kvx.kvx_conn_prefill(conn, 9, 0, [3], n_tokens=60, last_chunk=True, now_us=4)
    assert kvx.kvx_conn_poll(conn, 4) == [(9, 0, kvx.KVX_CONN_READY)]
    info = kvx.kvx_conn_get(conn, 9)
    assert (info["n_chunks"], info["n_src"], info["n_tokens"]) == (3, 4, 60)
    assert list(kvx.kvx_conn_ids(conn, 9)[0]) == [0, 1, 2, 3]
    assert status_of(kvx.kvx_conn_prefill, conn, 9, 0, [4], 64, True, 5) == kvx.KVX_EINVAL


def test_chunks_without_registration_defer_only_after_the_last(conn):
    kvx.kvx_conn_prefill(conn, 10, 0, [0], 16, False, now_us=0)
    assert state(conn, 10) == kvx.KVX_CONN_WAITING
    assert kvx.kvx_conn_poll(conn, 100 * S) == []                  # no defer clock before the last chunk
    kvx.kvx_conn_prefill(conn, 10, 0, [1], 32, True, now_us=100 * S)
    assert state(conn, 10) == kvx.KVX_CONN_DEFERRED
    assert kvx.kvx_conn_poll(conn, 160 * S - 1) == []
    assert kvx.kvx_conn_poll(conn, 160 * S) == [(10, 0, kvx.KVX_CONN_EXPIRED)]


def test_seal_fixes_the_expected_count_at_the_writes_queued(conn):
    # a hybrid model queues fewer writes than it has layers: completion follows the queued count
    kvx.kvx_conn_register(conn, 11, 0, [0, 1], now_us=0)
    kvx.kvx_conn_prefill(conn, 11, 0, [5, 6], 32, True, now_us=0)
    kvx.kvx_conn_start(conn, 11, 0, now_us=0)
    kvx.kvx_conn_write_issued(conn, 11, 0, 0, 2)
    kvx.kvx_conn_write_done(conn, 11, 0, 0, [DONE, DONE])
    kvx.kvx_conn_write_issued(conn, 11, 0, 0, 1)
    kvx.kvx_conn_write_done(conn, 11, 0, 0, [DONE])
    assert state(conn, 11) == kvx.KVX_CONN_IN_FLIGHT               # not sealed: more may come
    kvx.kvx_conn_write_done(conn, 11, 0, 0, [DONE])
    assert state(conn, 11) == kvx.KVX_CONN_IN_FLIGHT
    kvx.kvx_conn_seal(conn, 11, 0, 0)
    info = kvx.kvx_conn_get(conn, 11)
    assert (info["state"], info["writes_expected"], info["writes_done"], info["ranks_sealed"]) == \
        (kvx.KVX_CONN_DONE, 3, 3, 1)
    assert kvx.kvx_conn_poll(conn, 1)[-1] == (11, 0, kvx.KVX_CONN_DONE)


def test_seal_before_the_reports_and_over_reporting(conn):
    kvx.kvx_conn_register(conn, 12, 0, [0], now_us=0)
    kvx.kvx_conn_prefill(conn, 12, 0, [5], 16, True, now_us=0)
    kvx.kvx_conn_start(conn, 12, 0, now_us=0)
    kvx.kvx_conn_write_issued(conn, 12, 0, 0, 2)
    kvx.kvx_conn_seal(conn, 12, 0, 0)
    kvx.kvx_conn_seal(conn, 12, 0, 0)                              # a second seal changes nothing
    assert status_of(kvx.kvx_conn_write_issued, conn, 12, 0, 0, 1) == kvx.KVX_EINVAL
    kvx.kvx_conn_write_done(conn, 12, 0, 0, [DONE])
    assert state(conn, 12) == kvx.KVX_CONN_IN_FLIGHT
    kvx.kvx_conn_write_done(conn, 12, 0, 0, [DONE])
    assert state(conn, 12) == kvx.KVX_CONN_DONE
    assert status_of(kvx.kvx_conn_write_done, conn, 12, 0, 0, [DONE]) == kvx.KVX_EINVAL
    assert kvx.kvx_conn_get(conn, 12)["writes_done"] == 2


def test_a_rank_may_not_report_more_than_it_queued_before_sealing(conn):
    kvx.kvx_conn_register(conn, 13, 0, [0], now_us=0)
    kvx.kvx_conn_prefill(conn, 13, 0, [5], 16, True, now_us=0)
    kvx.kvx_conn_start(conn, 13, 0, now_us=0)
    assert status_of(kvx.kvx_conn_write_done, conn, 13, 0, 0, [DONE]) == kvx.KVX_EINVAL


def test_zero_writes_sealed_completes_at_once(conn):
    kvx.kvx_conn_register(conn, 14, 0, [], now_us=0)                # nothing to move (full local hit)
    kvx.kvx_conn_prefill(conn, 14, 0, [], 0, True, now_us=0)
    kvx.kvx_conn_start(conn, 14, 0, now_us=0)
    kvx.kvx_conn_seal(conn, 14, 0, 0)
    assert state(conn, 14) == kvx.KVX_CONN_DONE


def test_every_rank_must_seal_and_report():
    # consumer TP 8 over producer TP 2: 8 / 2 = 4 acknowledgements complete a request
    c = kvx.kvx_conn_create(n_ranks=4)
    kvx.kvx_conn_register(c, 1, 0, [0, 1], now_us=0)
    kvx.kvx_conn_prefill(c, 1, 0, [2, 3], 32, True, now_us=0)
    kvx.kvx_conn_start(c, 1, 0, now_us=0)
    for r in range(4):
        kvx.kvx_conn_write_issued(c, 1, 0, r, 1)
    for r in (3, 1, 0):
        kvx.kvx_conn_seal(c, 1, 0, r)
        kvx.kvx_conn_write_done(c, 1, 0, r, [DONE])
        assert state(c, 1) == kvx.KVX_CONN_IN_FLIGHT
    kvx.kvx_conn_write_done(c, 1, 0, 2, [DONE])
    assert state(c, 1) == kvx.KVX_CONN_IN_FLIGHT                   # rank 2 has not sealed
    kvx.kvx_conn_seal(c, 1, 0, 2)
    assert state(c, 1) == kvx.KVX_CONN_DONE
    assert status_of(kvx.kvx_conn_seal, c, 1, 0, 4) == kvx.KVX_EINVAL
    kvx.kvx_conn_destroy(c)


def test_batch_state_is_decided_over_all_layers(conn):
    kvx.kvx_conn_register(conn, 15, 0, [50, 51, 52, 53], now_us=0)
    kvx.kvx_conn_prefill(conn, 15, 0, [0, 1, 2, 3], 64, True, now_us=0)
    kvx.kvx_conn_start(conn, 15, 0, now_us=0)
    kvx.kvx_conn_write_issued(conn, 15, 0, 0, 2)
    kvx.kvx_conn_seal(conn, 15, 0, 0)
    kvx.kvx_conn_write_done(conn, 15, 0, 0, [DONE, DONE, DONE])
    # a middle layer failed; the last one reported is DONE
    kvx.kvx_conn_write_done(conn, 15, 0, 0, [DONE, FAILED, DONE], failed_blocks=[52, 53])
    info = kvx.kvx_conn_get(conn, 15)
    assert info["state"] == kvx.KVX_CONN_FAILED and info["writes_failed"] == 1
    assert list(kvx.kvx_conn_load_errors(conn, 15)) == [52, 53]
    assert info["first_error"] == 2                                 # tokens from block 2 on are recomputed


def test_a_failed_write_without_block_list_fails_every_registered_block(conn):
    kvx.kvx_conn_register(conn, 16, 0, [7, 3, 9], now_us=0)
    kvx.kvx_conn_prefill(conn, 16, 0, [0, 1, 2], 48, True, now_us=0)
    kvx.kvx_conn_start(conn, 16, 0, now_us=0)
    kvx.kvx_conn_write_issued(conn, 16, 0, 0, 2)
    kvx.kvx_conn_write_done(conn, 16, 0, 0, [FAILED])
    kvx.kvx_conn_write_done(conn, 16, 0, 0, [FAILED], failed_blocks=[3])   # no duplicates
    kvx.kvx_conn_seal(conn, 16, 0, 0)
    assert list(kvx.kvx_conn_load_errors(conn, 16)) == [7, 3, 9]
    info = kvx.kvx_conn_get(conn, 16)
    assert (info["state"], info["n_load_errors"], info["first_error"], info["writes_failed"]) == \
        (kvx.KVX_CONN_FAILED, 3, 0, 2)


def test_pending_layers_are_not_a_finished_write(conn):
    kvx.kvx_conn_register(conn, 17, 0, [0], now_us=0)
    kvx.kvx_conn_prefill(conn, 17, 0, [0], 16, True, now_us=0)
    kvx.kvx_conn_start(conn, 17, 0, now_us=0)
    kvx.kvx_conn_write_issued(conn, 17, 0, 0, 1)
    for bad in ([DONE, PENDING], [IDLE], [FAILED, PENDING], [DONE, 9]):
        assert status_of(kvx.kvx_conn_write_done, conn, 17, 0, 0, bad) == kvx.KVX_EINVAL
    info = kvx.kvx_conn_get(conn, 17)
    assert (info["writes_done"], info["writes_failed"], info["n_load_errors"]) == (0, 0, 0)


def test_release_drops_pending_events_and_deadlines(conn):
    kvx.kvx_conn_prefill(conn, 18, 0, [0], 16, True, now_us=0)
    kvx.kvx_conn_register(conn, 19, 0, [0], now_us=0)
    kvx.kvx_conn_prefill(conn, 19, 0, [1], 16, True, now_us=0)
    assert kvx.kvx_conn_size(conn) == 2
    kvx.kvx_conn_release(conn, 18)
    kvx.kvx_conn_release(conn, 19)
    kvx.kvx_conn_release(conn, 12345)                                # unknown: a no-op
    assert kvx.kvx_conn_size(conn) == 0
    assert kvx.kvx_conn_poll(conn, 1000 * S) == []
    # the same id and attempt afterwards is a new record with fresh deadlines
    kvx.kvx_conn_prefill(conn, 18, 0, [0], 16, True, now_us=1000 * S)
    assert kvx.kvx_conn_poll(conn, 1059 * S) == []
    assert kvx.kvx_conn_poll(conn, 1060 * S) == [(18, 0, kvx.KVX_CONN_EXPIRED)]
    assert status_of(kvx.kvx_conn_get, conn, 19) == kvx.KVX_EINVAL


def test_poll_hands_out_events_in_order_up_to_cap(conn):
    for rid in range(10):
        kvx.kvx_conn_register(conn, rid, 0, [rid], now_us=rid)
    for rid in reversed(range(10)):
        kvx.kvx_conn_prefill(conn, rid, 0, [rid], 16, True, now_us=100)
    first = kvx.kvx_conn_poll(conn, 100, cap=4)
    rest = kvx.kvx_conn_poll(conn, 100, cap=100)
    assert [e[0] for e in first + rest] == list(reversed(range(10)))
    assert len(first) == 4 and all(e[2] == kvx.KVX_CONN_READY for e in first + rest)


def test_argument_checks():
    bad_cfgs = [dict(defer_timeout_us=-1), dict(n_ranks=-2), dict(recv_abort_timeout_us=-5), dict(n_ranks=65537)]
    for cfg in bad_cfgs:
        with pytest.raises(kvx.KvxError) as ei:
            kvx.kvx_conn_create(**cfg)
        assert ei.value.status == kvx.KVX_EINVAL
    c = kvx.kvx_conn_create()
    assert status_of(kvx.kvx_conn_register, c, 1, -1, [0], 0) == kvx.KVX_EINVAL
    assert status_of(kvx.kvx_conn_prefill, c, 1, 0, [0], -3, True, 0) == kvx.KVX_EINVAL
    assert status_of(kvx.kvx_conn_get, c, 404) == kvx.KVX_EINVAL
    assert status_of(kvx.kvx_conn_start, c, 404, 0, 0) == kvx.KVX_EINVAL
    kvx.kvx_conn_register(c, 1, 0, [0, 1, 2], now_us=0)
    assert status_of(kvx.kvx_conn_write_issued, c, 1, 0, 0, 1) == kvx.KVX_EINVAL   # not in flight
    assert status_of(kvx.kvx_conn_start, c, 1, 1, 0) == kvx.KVX_EINVAL             # wrong attempt
    # an id buffer that is too small is refused, not overrun
    small = np.full(3, -7, np.int32)
    st = kvx._lib.kvx_conn_ids(c.handle, 1, None, 0, small.ctypes.data_as(kvx._P(kvx.c_i32)), 2)
    assert st == kvx.KVX_ERANGE and (small == -7).all()
    kvx.kvx_conn_destroy(c)
    kvx.kvx_conn_destroy(c)                                         # the binding makes a second destroy a no-op


# ---------------------------------------------------------------------------------------------
# randomized interleavings: invariants that follow from the protocol, whatever the order
# ---------------------------------------------------------------------------------------------

def test_random_interleavings_keep_the_protocol_invariants():
    rng = random.Random(20261202)
    defer, transfer, abort = 50, 80, 400
    c = kvx.kvx_conn_create(defer_timeout_us=defer, transfer_timeout_us=transfer, recv_abort_timeout_us=abort,
                            n_ranks=2)
    n_req = 200
    # per request: ordered list of (time, action) -- chunks, a registration (maybe resent), maybe a retry
    plan = []
    for rid in range(n_req):
        t_reg = rng.randrange(0, 300)
        n_chunks = rng.randrange(1, 4)
        t_chunks = sorted(rng.randrange(0, 300) for _ in range(n_chunks))
        acts = [(t_reg, "reg"), (t_reg + rng.randrange(0, 5), "reg")] if rng.random() < 0.9 else []
        acts += [(t, "chunk", i == n_chunks - 1) for i, t in enumerate(t_chunks)]
        plan.append(sorted(acts, key=lambda a: a[0]))
    ops = sorted(((a[0], rid, a) for rid, acts in enumerate(plan) for a in acts), key=lambda x: (x[0], x[1]))
    seen = {rid: [] for rid in range(n_req)}
    registered, last_chunk_at, reg_at = set(), {}, {}
    started = {}

    def drain(now):
        for rid, att, st in kvx.kvx_conn_poll(c, now):
            assert att == 0
            seen[rid].append((now, st))

    now = 0
    for t, rid, a in ops:
        while now < t:                                              # advance the fake clock in small steps
            now += 1
            drain(now)
            # the producer side starts and finishes READY requests at random moments
            for r in range(n_req):
                info = kvx.kvx_conn_get(c, r) if r in registered or r in last_chunk_at else None
                if info and info["state"] == kvx.KVX_CONN_READY and rng.random() < 0.3:
                    kvx.kvx_conn_start(c, r, 0, now)
                    started[r] = now
                    for k in range(2):
                        kvx.kvx_conn_write_issued(c, r, 0, k, 1)
                        kvx.kvx_conn_seal(c, r, 0, k)
                elif info and info["state"] == kvx.KVX_CONN_IN_FLIGHT and rng.random() < 0.05:
                    k = 0 if info["writes_done"] == 0 else 1
                    kvx.kvx_conn_write_done(c, r, 0, k, [DONE, FAILED if rng.random() < 0.1 else DONE])
        if a[1] == "reg":
            st = status_of(kvx.kvx_conn_register, c, rid, 0, [rid, rid + 1000], now)
            assert st in (kvx.KVX_OK, kvx.KVX_ETIMEDOUT)
            if st == kvx.KVX_OK and rid not in registered:
                registered.add(rid)
                reg_at[rid] = now
        else:
            kvx.kvx_conn_prefill(c, rid, 0, [rid], 16, a[2], now)
            if a[2]:
                last_chunk_at[rid] = now
    end = now + abort + transfer + defer + 10
    drain(end)

    terminal = {kvx.KVX_CONN_DONE, kvx.KVX_CONN_FAILED, kvx.KVX_CONN_EXPIRED, kvx.KVX_CONN_TIMED_OUT,
                kvx.KVX_CONN_ABORTED}
    for rid in range(n_req):
        ev = seen[rid]
        states = [s for _, s in ev]
        final = kvx.kvx_conn_get(c, rid)["state"]
        # at most one READY; at most one terminal event, and it is the final state
        assert states.count(kvx.KVX_CONN_READY) <= 1
        assert sum(s in terminal for s in states) <= 1
        if any(s in terminal for s in states):
            assert states[-1] == final
        if kvx.KVX_CONN_READY in states:
            t_ready = ev[states.index(kvx.KVX_CONN_READY)][0]
            # READY only once both halves are in, and no earlier than the later of the two
            assert rid in registered and rid in last_chunk_at
            assert t_ready >= max(reg_at[rid], last_chunk_at[rid])
        if final == kvx.KVX_CONN_EXPIRED:
            assert rid in last_chunk_at and rid not in registered
        if final in (kvx.KVX_CONN_DONE, kvx.KVX_CONN_FAILED):
            info = kvx.kvx_conn_get(c, rid)
            assert info["writes_done"] == info["writes_expected"] == 2 and info["ranks_sealed"] == 2
            assert (final == kvx.KVX_CONN_FAILED) == (info["writes_failed"] > 0)
        if final == kvx.KVX_CONN_TIMED_OUT:
            assert rid in started
        if rid in registered:
            assert final in terminal                                # every registered request ends
    finals = {kvx.kvx_conn_get(c, rid)["state"] for rid in range(n_req)}
    assert terminal <= finals                                       # the draw reaches every outcome
    kvx.kvx_conn_destroy(c)


def test_threads_driving_both_sides_concurrently():
    """The main loop (registrations, chunks, polls) and a transfer thread (start, writes, seal) share
    one connector; ctypes releases the GIL, so the calls really overlap."""
    c = kvx.kvx_conn_create(n_ranks=1)
    n = 3000
    ready = []
    lock = threading.Lock()
    stop = threading.Event()

    def transfer_thread():
        done = 0
        while done < n and not stop.is_set():
            with lock:
                batch, ready[:] = list(ready), []
            for rid in batch:
                kvx.kvx_conn_start(c, rid, 0, 0)
                kvx.kvx_conn_write_issued(c, rid, 0, 0, 2)
                kvx.kvx_conn_write_done(c, rid, 0, 0, [DONE])
                kvx.kvx_conn_seal(c, rid, 0, 0)
                kvx.kvx_conn_write_done(c, rid, 0, 0, [DONE, DONE])
                done += 1

    th = threading.Thread(target=transfer_thread)
    th.start()
    finished = 0
    try:
        for rid in range(n):
            if rid % 2:
                kvx.kvx_conn_register(c, rid, 0, [rid], 0)
                kvx.kvx_conn_prefill(c, rid, 0, [rid], 16, True, 0)
            else:
                kvx.kvx_conn_prefill(c, rid, 0, [rid], 16, True, 0)
                kvx.kvx_conn_register(c, rid, 0, [rid], 0)
            for r, _, st in kvx.kvx_conn_poll(c, 0, cap=64):
                if st == kvx.KVX_CONN_READY:
                    with lock:
                        ready.append(r)
                elif st == kvx.KVX_CONN_DONE:
                    finished += 1
                    kvx.kvx_conn_release(c, r)
        deadline = time.monotonic() + 60
        while finished < n and time.monotonic() < deadline:
            time.sleep(0.0005)
            for r, _, st in kvx.kvx_conn_poll(c, 0, cap=256):
                if st == kvx.KVX_CONN_READY:
                    with lock:
                        ready.append(r)
                elif st == kvx.KVX_CONN_DONE:
                    finished += 1
                    kvx.kvx_conn_release(c, r)
    finally:
        stop.set() if finished != n else None
        th.join(timeout=60)
    assert finished == n and kvx.kvx_conn_size(c) == 0
    kvx.kvx_conn_destroy(c)
