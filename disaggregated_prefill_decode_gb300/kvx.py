"""Thin ctypes binding of the kvx C-ABI (include/kvx.h): same names, argument marshalling only.

Every operation runs in libkvx.so (hand-written CUDA for sm_103a). There is no fallback: importing
this module raises if the library has not been built (``__graft_entry__.build()`` or
``python disaggregated_prefill_decode_gb300/build.py``). PyTorch is used by callers only to own device
memory and streams; this module accepts torch tensors / streams / events or raw integer handles.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvx.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"kvx CUDA library not built: {_LIB_PATH} is missing (run __graft_entry__.build())")
_lib = ctypes.CDLL(_LIB_PATH)

c_i32, c_i64, c_u64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p

KVX_OK, KVX_EINVAL, KVX_ERANGE, KVX_EOVERLAP, KVX_EUNSUPPORTED, KVX_ENOMEM, KVX_ECUDA, KVX_ETIMEDOUT, \
    KVX_EFAILED = range(9)
KVX_LAYER_IDLE, KVX_LAYER_PENDING, KVX_LAYER_DONE, KVX_LAYER_FAILED = range(4)


class kvx_pool(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("n_planes", c_i32), ("n_shards", c_i32), ("heads_per_shard", c_i32),
                ("head_dim", c_i32), ("elem_bytes", c_i32), ("block_size", c_i32), ("layout", c_i32),
                ("n_blocks", c_i64), ("base", ctypes.POINTER(c_vp))]


KVX_LAYOUT_NHD, KVX_LAYOUT_HND = 0, 1


class kvx_request(ctypes.Structure):
    _fields_ = [("req_id", c_i64), ("n_tokens", c_i64), ("src_block_ids", ctypes.POINTER(c_i32)), ("n_src", c_i32),
                ("dst_block_ids", ctypes.POINTER(c_i32)), ("n_dst", c_i32)]


class kvx_plan_opts(ctypes.Structure):
    _fields_ = [("tile_bytes", c_i32), ("threads", c_i32), ("flags", c_i32), ("kernel", c_i32), ("ctas_per_sm", c_i32),
                ("lanes", c_i32), ("bulk_stages", c_i32), ("layers_per_launch", c_i32), ("max_ctas", c_i32)]


KVX_PLAN_TIMING = 1
KVX_KERNEL_AUTO, KVX_KERNEL_TILE, KVX_KERNEL_PERSIST, KVX_KERNEL_BULK, KVX_KERNEL_TENSOR, KVX_KERNEL_STAGED = range(6)


class kvx_plan_info(ctypes.Structure):
    _fields_ = [("n_runs", c_i64), ("n_tiles", c_i64), ("bytes_per_layer", c_i64), ("vec_bytes", c_i32),
                ("strided", c_i32), ("n_layers", c_i32), ("n_planes", c_i32), ("width", c_i32),
                ("tile_bytes", c_i32), ("kernel", c_i32), ("threads", c_i32), ("lanes", c_i32), ("bulk_stages", c_i32),
                ("src_pitch", c_i64), ("dst_pitch", c_i64), ("src_head_pitch", c_i64), ("dst_head_pitch", c_i64)]


class kvx_match_opts(ctypes.Structure):
    _fields_ = [("flags", c_i32), ("reserved0", c_i32), ("expiry", c_vp), ("now", c_i64), ("reserved", c_i64 * 4)]


KVX_MATCH_FILL_HOLES, KVX_MATCH_KEEP_LAST, KVX_MATCH_TEST_SCAN_STALL = 1, 2, 256


class kvx_match_result(ctypes.Structure):
    _fields_ = [("local_hit_blocks", c_i32), ("remote_hit_blocks", c_i32), ("missing_tokens", c_i32),
                ("push", c_i32), ("dst_start", c_i64)]


MATCH_RESULT_DTYPE = np.dtype([("local_hit_blocks", "<i4"), ("remote_hit_blocks", "<i4"), ("missing_tokens", "<i4"),
                               ("push", "<i4"), ("dst_start", "<i8")])
assert MATCH_RESULT_DTYPE.itemsize == ctypes.sizeof(kvx_match_result)

class kvx_conn_config(ctypes.Structure):
    _fields_ = [("defer_timeout_us", c_i64), ("transfer_timeout_us", c_i64), ("recv_abort_timeout_us", c_i64),
                ("n_ranks", c_i32), ("reserved", c_i32)]


class kvx_conn_event(ctypes.Structure):
    _fields_ = [("req_id", c_i64), ("attempt", c_i32), ("state", c_i32)]


class kvx_conn_info(ctypes.Structure):
    _fields_ = [("attempt", c_i32), ("state", c_i32), ("n_tokens", c_i64), ("n_src", c_i32), ("n_dst", c_i32),
                ("n_chunks", c_i32), ("ranks_sealed", c_i32), ("writes_issued", c_i64), ("writes_expected", c_i64),
                ("writes_done", c_i64), ("writes_failed", c_i64), ("n_load_errors", c_i32), ("first_error", c_i32)]


KVX_CONN_WAITING, KVX_CONN_DEFERRED, KVX_CONN_READY, KVX_CONN_IN_FLIGHT, KVX_CONN_DONE, KVX_CONN_FAILED, \
    KVX_CONN_EXPIRED, KVX_CONN_TIMED_OUT, KVX_CONN_ABORTED = range(9)

TILE_DTYPE = np.dtype([("src_off", "<i8"), ("dst_off", "<i8"), ("n", "<i4"), ("src_shard", "<i4"),
                       ("dst_shard", "<i4"), ("heads", "<i4")])

_P = ctypes.POINTER
_sig = {
    "kvx_plan": (c_i32, [_P(kvx_pool), _P(kvx_pool), _P(kvx_request), c_i32, _P(c_vp)]),
    "kvx_plan_ex": (c_i32, [_P(kvx_pool), _P(kvx_pool), _P(kvx_request), c_i32, _P(kvx_plan_opts), _P(c_vp)]),
    "kvx_plan_set_opts": (c_i32, [c_vp, _P(kvx_plan_opts)]),
    "kvx_plan_runs": (c_i32, [c_vp, _P(c_i64), _P(_P(c_i32)), _P(_P(c_i32)), _P(_P(c_i32))]),
    "kvx_plan_get_info": (c_i32, [c_vp, _P(kvx_plan_info)]),
    "kvx_plan_tiles": (c_i32, [c_vp, _P(c_i64), _P(c_vp)]),
    "kvx_push_layer": (c_i32, [c_vp, c_i32, c_vp, c_vp]),
    "kvx_push_layers": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp]),
    "kvx_push_layer_notify": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "kvx_sync": (c_i32, [c_vp, c_i64]),
    "kvx_plan_layer_states": (c_i32, [c_vp, _P(c_i32), c_i32]),
    "kvx_plan_push_times": (c_i32, [c_vp, _P(ctypes.c_float), _P(ctypes.c_float), c_i32, _P(c_i32)]),
    "kvx_plan_push_times_ns": (c_i32, [c_vp, _P(c_i64), _P(c_i64), c_i32, _P(c_i32)]),
    "kvx_plan_inject_failure": (c_i32, [c_vp, c_i32]),
    "kvx_plan_inject_stall": (c_i32, [c_vp, c_i32]),
    "kvx_plan_destroy": (c_i32, [c_vp]),
    "kvx_status_str": (ctypes.c_char_p, [c_i32]),
    "kvx_last_error": (ctypes.c_char_p, []),
    "kvx_block_hashes": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "kvx_block_hashes_ex": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "kvx_table_build": (c_i32, [c_vp, c_vp, c_i64, c_vp, _P(c_vp)]),
    "kvx_table_lookup": (c_i32, [c_vp, c_vp, c_i64, c_vp, c_vp]),
    "kvx_table_destroy": (c_i32, [c_vp]),
    "kvx_match_prefix": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_i64,
                                 _P(kvx_pool), _P(kvx_pool), c_vp, _P(c_vp), c_vp]),
    "kvx_match_prefix_ex": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_i64,
                                    _P(kvx_pool), _P(kvx_pool), c_vp, c_vp, _P(c_vp), c_vp]),
    "kvx_match_prefix_static": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_i64, c_vp, c_vp]),
    "kvx_conn_create": (c_i32, [_P(kvx_conn_config), _P(c_vp)]),
    "kvx_conn_destroy": (c_i32, [c_vp]),
    "kvx_conn_register": (c_i32, [c_vp, c_i64, c_i32, _P(c_i32), c_i32, c_i64]),
    "kvx_conn_prefill": (c_i32, [c_vp, c_i64, c_i32, _P(c_i32), c_i32, c_i64, c_i32, c_i64]),
    "kvx_conn_poll": (c_i32, [c_vp, c_i64, _P(kvx_conn_event), c_i32, _P(c_i32)]),
    "kvx_conn_get": (c_i32, [c_vp, c_i64, _P(kvx_conn_info)]),
    "kvx_conn_ids": (c_i32, [c_vp, c_i64, _P(c_i32), c_i32, _P(c_i32), c_i32]),
    "kvx_conn_start": (c_i32, [c_vp, c_i64, c_i32, c_i64]),
    "kvx_conn_write_issued": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32]),
    "kvx_conn_seal": (c_i32, [c_vp, c_i64, c_i32, c_i32]),
    "kvx_conn_write_done": (c_i32, [c_vp, c_i64, c_i32, c_i32, _P(c_i32), c_i32, _P(c_i32), c_i32, c_i64]),
    "kvx_conn_load_errors": (c_i32, [c_vp, c_i64, _P(c_i32), c_i32, _P(c_i32)]),
    "kvx_conn_release": (c_i32, [c_vp, c_i64]),
    "kvx_conn_size": (c_i64, [c_vp]),
    "kvx_version": (ctypes.c_char_p, []),
    "kvx_launch_count": (c_i64, []),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


class KvxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvx_status_str(status)}: {kvx_last_error()}")


def _check(st: int, where: str) -> int:
    if st != KVX_OK:
        raise KvxError(st, where)
    return st


def kvx_status_str(status: int) -> str:
    return _lib.kvx_status_str(status).decode()


def kvx_last_error() -> str:
    return _lib.kvx_last_error().decode()


def kvx_version() -> str:
    return _lib.kvx_version().decode()


def kvx_launch_count() -> int:
    return int(_lib.kvx_launch_count())


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------

def _ptr(x) -> int:
    """Device pointer of a torch tensor, or an int passed through. None -> 0."""
    if x is None:
        return 0
    if isinstance(x, (int, np.integer)):
        return int(x)
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _event(e) -> int:
    if e is None:
        return 0
    if isinstance(e, int):
        return e
    return int(e.cuda_event)


class Pool:
    """A kvx_pool plus the pointer table it references. `geom` has the kvx_pool count fields;
    `buffers` lists one device buffer (torch tensor or pointer) per (layer, plane, shard)."""

    def __init__(self, geom, buffers: Sequence):
        n = geom.n_layers * geom.n_planes * geom.n_shards
        if len(buffers) != n:
            raise ValueError(f"pool needs {n} buffers, got {len(buffers)}")
        self.geom = geom
        self.buffers = list(buffers)
        self._ptrs = (c_vp * max(n, 1))(*[_ptr(b) for b in buffers])
        self.struct = kvx_pool(geom.n_layers, geom.n_planes, geom.n_shards, geom.heads_per_shard, geom.head_dim,
                               geom.elem_bytes, geom.block_size, getattr(geom, "layout", 0), geom.n_blocks,
                               ctypes.cast(self._ptrs, _P(c_vp)))


class Plan:
    """Owns a kvx_plan_t handle; call kvx_plan_destroy (or use `with`) to free it."""

    def __init__(self, handle: int, n_layers: int):
        self.handle = handle
        self.n_layers = n_layers

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        kvx_plan_destroy(self)


class Table:
    def __init__(self, handle: int):
        self.handle = handle


def _requests(reqs) -> tuple:
    """reqs: iterable of (n_tokens, src_ids, dst_ids) or (n_tokens, src_ids, dst_ids, req_id)."""
    keep, arr = [], []
    for i, r in enumerate(reqs):
        n_tok, sids, dids = int(r[0]), np.ascontiguousarray(r[1], np.int32), np.ascontiguousarray(r[2], np.int32)
        rid = int(r[3]) if len(r) > 3 else i
        keep += [sids, dids]
        arr.append(kvx_request(rid, n_tok, sids.ctypes.data_as(_P(c_i32)), len(sids),
                               dids.ctypes.data_as(_P(c_i32)), len(dids)))
    n = len(arr)
    carr = (kvx_request * max(n, 1))(*arr)
    return carr, n, keep


def _h(plan) -> int:
    return plan.handle if isinstance(plan, Plan) else int(plan)


# ---------------------------------------------------------------------------------------------
# C-ABI calls
# ---------------------------------------------------------------------------------------------

def kvx_plan(src: Pool, dst: Pool, requests: Iterable) -> Plan:
    return kvx_plan_ex(src, dst, requests, None)


_OPT_KEYS = ("tile_bytes", "threads", "flags", "kernel", "ctas_per_sm", "lanes", "bulk_stages", "layers_per_launch",
             "max_ctas")


def _opts(opts: dict) -> kvx_plan_opts:
    unknown = set(opts) - set(_OPT_KEYS)
    if unknown:
        raise ValueError(f"unknown plan options {sorted(unknown)}")
    return kvx_plan_opts(*(int(opts.get(k, 0)) for k in _OPT_KEYS))


def kvx_plan_ex(src: Pool, dst: Pool, requests: Iterable, opts: Optional[dict] = None) -> Plan:
    carr, n, _keep = _requests(requests)
    out = c_vp()
    o = _opts(opts) if opts else None
    st = _lib.kvx_plan_ex(ctypes.byref(src.struct), ctypes.byref(dst.struct), carr, n,
                          ctypes.byref(o) if o is not None else None, ctypes.byref(out))
    _check(st, "kvx_plan")
    return Plan(out.value, src.geom.n_layers)


def kvx_plan_set_opts(plan, opts: dict) -> None:
    o = _opts(opts)
    _check(_lib.kvx_plan_set_opts(_h(plan), ctypes.byref(o)), "kvx_plan_set_opts")


def kvx_plan_runs(plan) -> tuple:
    n = c_i64()
    s, d, t = _P(c_i32)(), _P(c_i32)(), _P(c_i32)()
    _check(_lib.kvx_plan_runs(_h(plan), ctypes.byref(n), ctypes.byref(s), ctypes.byref(d), ctypes.byref(t)),
           "kvx_plan_runs")
    k = n.value
    if k == 0:
        z = np.zeros(0, np.int32)
        return z, z.copy(), z.copy()
    return (np.ctypeslib.as_array(s, (k,)).copy(), np.ctypeslib.as_array(d, (k,)).copy(),
            np.ctypeslib.as_array(t, (k,)).copy())


def kvx_plan_get_info(plan) -> dict:
    info = kvx_plan_info()
    _check(_lib.kvx_plan_get_info(_h(plan), ctypes.byref(info)), "kvx_plan_get_info")
    return {f: getattr(info, f) for f, _ in kvx_plan_info._fields_}


def kvx_plan_tiles(plan) -> np.ndarray:
    """Copy of a host-built plan's tile table (structured array of TILE_DTYPE)."""
    n = c_i64()
    p = c_vp()
    _check(_lib.kvx_plan_tiles(_h(plan), ctypes.byref(n), ctypes.byref(p)), "kvx_plan_tiles")
    if n.value == 0:
        return np.zeros(0, TILE_DTYPE)
    raw = (ctypes.c_uint8 * (32 * n.value)).from_address(p.value)
    return np.frombuffer(bytes(raw), TILE_DTYPE).copy()


def kvx_push_layer(plan, layer: int, stream=None, ready=None) -> None:
    _check(_lib.kvx_push_layer(_h(plan), layer, _stream(stream), _event(ready)), "kvx_push_layer")


def kvx_push_layers(plan, layer_begin: int, layer_end: int, stream=None, ready=None) -> None:
    _check(_lib.kvx_push_layers(_h(plan), layer_begin, layer_end, _stream(stream), _event(ready)), "kvx_push_layers")


def kvx_push_layer_notify(plan, layer_begin: int, layer_end: int, stream, ready, done) -> None:
    _check(_lib.kvx_push_layer_notify(_h(plan), layer_begin, layer_end, _stream(stream), _event(ready), _event(done)),
           "kvx_push_layer_notify")


def kvx_sync(plan, timeout_us: int = -1) -> int:
    """Returns KVX_OK, KVX_ETIMEDOUT or KVX_EFAILED; raises on any other status."""
    st = _lib.kvx_sync(_h(plan), int(timeout_us))
    if st not in (KVX_OK, KVX_ETIMEDOUT, KVX_EFAILED):
        raise KvxError(st, "kvx_sync")
    return st


def kvx_plan_push_times(plan, cap: int = 4096) -> tuple:
    """(start_us, end_us) of each push confirmed by the last kvx_sync, relative to the earliest start
    among them (timing plans; the kernels' own global-timer stamps)."""
    s, e = np.zeros(cap, np.float32), np.zeros(cap, np.float32)
    n = c_i32()
    _check(_lib.kvx_plan_push_times(_h(plan), s.ctypes.data_as(_P(ctypes.c_float)), e.ctypes.data_as(_P(ctypes.c_float)),
                                    cap, ctypes.byref(n)), "kvx_plan_push_times")
    k = min(n.value, cap)
    return s[:k].copy(), e[:k].copy()


def kvx_plan_push_times_ns(plan, cap: int = 4096) -> tuple:
    """(start_ns, end_ns) of the same pushes as raw readings of the GPU's global timer."""
    s, e = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
    n = c_i32()
    _check(_lib.kvx_plan_push_times_ns(_h(plan), s.ctypes.data_as(_P(c_i64)), e.ctypes.data_as(_P(c_i64)),
                                       cap, ctypes.byref(n)), "kvx_plan_push_times_ns")
    k = min(n.value, cap)
    return s[:k].copy(), e[:k].copy()


def kvx_plan_layer_states(plan) -> np.ndarray:
    out = np.zeros(plan.n_layers, np.int32)
    _check(_lib.kvx_plan_layer_states(_h(plan), out.ctypes.data_as(_P(c_i32)), plan.n_layers), "kvx_plan_layer_states")
    return out


def kvx_plan_inject_failure(plan, layer: int) -> None:
    _check(_lib.kvx_plan_inject_failure(_h(plan), layer), "kvx_plan_inject_failure")


def kvx_plan_inject_stall(plan, layer: int) -> None:
    _check(_lib.kvx_plan_inject_stall(_h(plan), layer), "kvx_plan_inject_stall")


def kvx_plan_destroy(plan) -> None:
    h = _h(plan)
    if h:
        _check(_lib.kvx_plan_destroy(h), "kvx_plan_destroy")
    if isinstance(plan, Plan):
        plan.handle = 0


def kvx_block_hashes(tokens, tok_off, n_sessions: int, block_size: int, out_hash, hash_off, stream=None) -> None:
    _check(_lib.kvx_block_hashes(_ptr(tokens), _ptr(tok_off), n_sessions, block_size, _ptr(out_hash), _ptr(hash_off),
                                 _stream(stream)), "kvx_block_hashes")


def kvx_block_hashes_ex(tokens, tok_off, n_sessions: int, block_size: int, parent, out_hash, hash_off,
                        stream=None) -> None:
    _check(_lib.kvx_block_hashes_ex(_ptr(tokens), _ptr(tok_off), n_sessions, block_size, _ptr(parent), _ptr(out_hash),
                                    _ptr(hash_off), _stream(stream)), "kvx_block_hashes_ex")


def kvx_table_build(keys, vals, n: int, stream=None) -> Table:
    out = c_vp()
    _check(_lib.kvx_table_build(_ptr(keys), _ptr(vals), n, _stream(stream), ctypes.byref(out)), "kvx_table_build")
    return Table(out.value)


def kvx_table_lookup(table: Table, keys, n: int, out_vals, stream=None) -> None:
    _check(_lib.kvx_table_lookup(table.handle, _ptr(keys), n, _ptr(out_vals), _stream(stream)), "kvx_table_lookup")


def kvx_table_destroy(table: Table) -> None:
    if table.handle:
        _check(_lib.kvx_table_destroy(table.handle), "kvx_table_destroy")
    table.handle = 0


def kvx_match_prefix(tokens, tok_off, n_sessions: int, block_size: int, table: Table, remote_hash, remote_blk,
                     rem_off, recompute_threshold_tokens: int, free_blocks, n_free: int, remote_pool: Optional[Pool],
                     local_pool: Optional[Pool], out, want_plan: bool = True, stream=None, flags: int = 0,
                     expiry=None, now: int = 0):
    """Returns (status, Plan or None). Status is KVX_OK or KVX_ENOMEM; other statuses raise. flags,
    expiry (device int64 per session) and now go to kvx_match_prefix_ex when given."""
    plan = c_vp()
    if flags or expiry is not None:
        o = kvx_match_opts(int(flags), 0, _ptr(expiry) or None, int(now))
        st = _lib.kvx_match_prefix_ex(_ptr(tokens), _ptr(tok_off), n_sessions, block_size, table.handle,
                                      _ptr(remote_hash), _ptr(remote_blk), _ptr(rem_off), recompute_threshold_tokens,
                                      _ptr(free_blocks), n_free, ctypes.byref(remote_pool.struct) if remote_pool else None,
                                      ctypes.byref(local_pool.struct) if local_pool else None, ctypes.byref(o),
                                      _ptr(out), ctypes.byref(plan) if want_plan else None, _stream(stream))
    else:
        st = _lib.kvx_match_prefix(_ptr(tokens), _ptr(tok_off), n_sessions, block_size, table.handle,
                                   _ptr(remote_hash), _ptr(remote_blk), _ptr(rem_off), recompute_threshold_tokens,
                                   _ptr(free_blocks), n_free, ctypes.byref(remote_pool.struct) if remote_pool else None,
                                   ctypes.byref(local_pool.struct) if local_pool else None, _ptr(out),
                                   ctypes.byref(plan) if want_plan else None, _stream(stream))
    if st not in (KVX_OK, KVX_ENOMEM):
        raise KvxError(st, "kvx_match_prefix")
    n_layers = remote_pool.geom.n_layers if remote_pool else 0
    return st, (Plan(plan.value, n_layers) if plan.value else None)


def kvx_match_prefix_static(tokens, tok_off, n_sessions: int, block_size: int, table: Table, remote_hash, rem_off,
                            recompute_threshold_tokens: int, n_free: int, out, stream=None) -> int:
    """Allocation-free match decision. Returns KVX_OK or KVX_ENOMEM; other statuses raise."""
    st = _lib.kvx_match_prefix_static(_ptr(tokens), _ptr(tok_off), n_sessions, block_size, table.handle,
                                      _ptr(remote_hash), _ptr(rem_off), recompute_threshold_tokens, n_free, _ptr(out),
                                      _stream(stream))
    if st not in (KVX_OK, KVX_ENOMEM):
        raise KvxError(st, "kvx_match_prefix_static")
    return st


# ---------------------------------------------------------------------------------------------
# connector state machine (host only)
# ---------------------------------------------------------------------------------------------

class Conn:
    def __init__(self, handle: int):
        self.handle = handle


def _conn(conn) -> int:
    if conn is None or not conn.handle:
        raise ValueError("connector was destroyed")
    return conn.handle


def _ids(a) -> tuple:
    """Host int32 id array (kept alive by the caller's reference) and its count."""
    a = np.ascontiguousarray(np.asarray(a if a is not None else [], dtype=np.int32))
    return a, a.ctypes.data_as(_P(c_i32)) if len(a) else None, len(a)


def kvx_conn_create(defer_timeout_us: int = 0, transfer_timeout_us: int = 0, recv_abort_timeout_us: int = 0,
                    n_ranks: int = 0) -> Conn:
    cfg = kvx_conn_config(defer_timeout_us, transfer_timeout_us, recv_abort_timeout_us, n_ranks, 0)
    h = c_vp()
    _check(_lib.kvx_conn_create(ctypes.byref(cfg), ctypes.byref(h)), "kvx_conn_create")
    return Conn(h.value)


def kvx_conn_destroy(conn: Conn) -> None:
    if conn.handle:
        _check(_lib.kvx_conn_destroy(conn.handle), "kvx_conn_destroy")
        conn.handle = None


def kvx_conn_register(conn: Conn, req_id: int, attempt: int, dst_ids, now_us: int) -> None:
    a, p, n = _ids(dst_ids)
    _check(_lib.kvx_conn_register(_conn(conn), req_id, attempt, p, n, now_us), "kvx_conn_register")


def kvx_conn_prefill(conn: Conn, req_id: int, attempt: int, src_ids, n_tokens: int, last_chunk: bool,
                     now_us: int) -> None:
    a, p, n = _ids(src_ids)
    _check(_lib.kvx_conn_prefill(_conn(conn), req_id, attempt, p, n, n_tokens, int(bool(last_chunk)), now_us),
           "kvx_conn_prefill")


def kvx_conn_poll(conn: Conn, now_us: int, cap: int = 1024) -> list:
    """Events as (req_id, attempt, state) tuples, in the order they happened."""
    out = (kvx_conn_event * max(cap, 1))()
    n = c_i32()
    _check(_lib.kvx_conn_poll(_conn(conn), now_us, out, cap, ctypes.byref(n)), "kvx_conn_poll")
    return [(out[i].req_id, out[i].attempt, out[i].state) for i in range(n.value)]


def kvx_conn_get(conn: Conn, req_id: int) -> dict:
    info = kvx_conn_info()
    _check(_lib.kvx_conn_get(_conn(conn), req_id, ctypes.byref(info)), "kvx_conn_get")
    return {name: getattr(info, name) for name, _ in kvx_conn_info._fields_}


def kvx_conn_ids(conn: Conn, req_id: int) -> tuple:
    info = kvx_conn_get(conn, req_id)
    src = np.zeros(max(info["n_src"], 1), np.int32)
    dst = np.zeros(max(info["n_dst"], 1), np.int32)
    _check(_lib.kvx_conn_ids(_conn(conn), req_id, src.ctypes.data_as(_P(c_i32)), info["n_src"],
                             dst.ctypes.data_as(_P(c_i32)), info["n_dst"]), "kvx_conn_ids")
    return src[:info["n_src"]], dst[:info["n_dst"]]


def kvx_conn_start(conn: Conn, req_id: int, attempt: int, now_us: int) -> None:
    _check(_lib.kvx_conn_start(_conn(conn), req_id, attempt, now_us), "kvx_conn_start")


def kvx_conn_write_issued(conn: Conn, req_id: int, attempt: int, rank: int, n_writes: int) -> None:
    _check(_lib.kvx_conn_write_issued(_conn(conn), req_id, attempt, rank, n_writes), "kvx_conn_write_issued")


def kvx_conn_seal(conn: Conn, req_id: int, attempt: int, rank: int) -> None:
    _check(_lib.kvx_conn_seal(_conn(conn), req_id, attempt, rank), "kvx_conn_seal")


def kvx_conn_write_done(conn: Conn, req_id: int, attempt: int, rank: int, layer_states, failed_blocks=None,
                        now_us: int = 0) -> None:
    s, ps, ns = _ids(layer_states)
    f, pf, nf = _ids(failed_blocks)
    _check(_lib.kvx_conn_write_done(_conn(conn), req_id, attempt, rank, ps, ns, pf, nf, now_us),
           "kvx_conn_write_done")


def kvx_conn_load_errors(conn: Conn, req_id: int) -> np.ndarray:
    n = c_i32()
    _check(_lib.kvx_conn_load_errors(_conn(conn), req_id, None, 0, ctypes.byref(n)), "kvx_conn_load_errors")
    out = np.zeros(max(n.value, 1), np.int32)
    _check(_lib.kvx_conn_load_errors(_conn(conn), req_id, out.ctypes.data_as(_P(c_i32)), n.value, ctypes.byref(n)),
           "kvx_conn_load_errors")
    return out[:n.value]


def kvx_conn_release(conn: Conn, req_id: int) -> None:
    _check(_lib.kvx_conn_release(_conn(conn), req_id), "kvx_conn_release")


def kvx_conn_size(conn: Conn) -> int:
    return int(_lib.kvx_conn_size(_conn(conn)))


def library_path() -> str:
    return _LIB_PATH
