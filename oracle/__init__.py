"""kvx oracle -- TEST INFRASTRUCTURE ONLY.

Python entry points over the plain C oracle in ``kvx_oracle.c`` (built with gcc into
``oracle/_build``). Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package; the kvx library never does, and it shares no code with it.

Functions and the passages they follow (see the C file for the full citations):
  push         -- "Push-based KV transfer" (spke.com 3844), Implementierungsdetails step 3; MoRIIO
                  notes section 6, rank mapping. Per-head byte copy, token by token.
  block_runs   -- same article, Threading-Modell; MoRIIO notes section 6, memory registration and
  token_runs      offset calculation. Maximal contiguous runs, merged within a request.
  fnv1a64      -- FNV-1a as published by Fowler, Noll and Vo.
  block_hashes -- chained FNV-1a block hashes (parent hash, then the block's token ids).
  match        -- "Bidirectional KV transfer" (spke.com 3845), Figure 1 steps 4-6 and the KV recompute
                  threshold section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Iterable, List, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvx_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libkvx_oracle.so")

FNV64_OFFSET_BASIS = 14695981039346656037


def build(src: str = _SRC, out: str = LIB_PATH, extra_flags: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc (plain C99, -O2). Rebuilds only when the source is newer."""
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra_flags:
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-std=c99", "-O2", "-shared", "-fPIC", *extra_flags, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _Pool(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("n_planes", ctypes.c_int32), ("n_shards", ctypes.c_int32),
        ("heads_per_shard", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32), ("block_size", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("n_blocks", ctypes.c_int64), ("base", ctypes.POINTER(ctypes.c_void_p)),
    ]


_P = ctypes.c_void_p
_I32, _I64, _U64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64


class Oracle:
    """One loaded copy of the oracle library (tests may load a deliberately altered build)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_push.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Pool), _I32, _P, _P, _P]
        lib.oracle_push.restype = ctypes.c_int
        lib.oracle_block_runs.argtypes = [_I32, _P, _P, _P, _P, _P]
        lib.oracle_block_runs.restype = _I32
        lib.oracle_token_runs.argtypes = [_I64, _I32, _P, _I32, _P, _P, _P, _P]
        lib.oracle_token_runs.restype = _I64
        lib.oracle_fnv1a64.argtypes = [_P, _I64, _U64]
        lib.oracle_fnv1a64.restype = _U64
        lib.oracle_fnv64_offset_basis.argtypes = []
        lib.oracle_fnv64_offset_basis.restype = _U64
        lib.oracle_block_hashes.argtypes = [_P, _I64, _I32, _P]
        lib.oracle_block_hashes.restype = _I64
        lib.oracle_match.argtypes = [_I32, _P, _P, _I32, _P, _I64, _P, _P, _P, _I32, _P, _I64,
                                     _P, _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_match.restype = ctypes.c_int
        lib.oracle_match_ex.argtypes = [_I32, _P, _P, _I32, _P, _I64, _P, _P, _P, _I32, _P, _I64, _I32, _P, _I64,
                                        _P, _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_match_ex.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    # -- push -----------------------------------------------------------------------------------
    @staticmethod
    def _pool(geom, bufs: List[np.ndarray], keep: list) -> _Pool:
        n = geom.n_layers * geom.n_planes * geom.n_shards
        if len(bufs) != n:
            raise ValueError(f"expected {n} buffers, got {len(bufs)}")
        need = geom.n_blocks * geom.block_size * geom.heads_per_shard * geom.head_dim * geom.elem_bytes
        ptrs = (ctypes.c_void_p * n)()
        for i, b in enumerate(bufs):
            if b.dtype != np.uint8 or not b.flags["C_CONTIGUOUS"] or b.nbytes < need:
                raise ValueError("oracle buffers must be C-contiguous uint8 of the full pool size")
            ptrs[i] = b.ctypes.data
        keep.append(ptrs)
        return _Pool(geom.n_layers, geom.n_planes, geom.n_shards, geom.heads_per_shard, geom.head_dim,
                     geom.elem_bytes, geom.block_size, getattr(geom, "layout", 0), geom.n_blocks,
                     ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)))

    def push(self, src_geom, src_bufs, dst_geom, dst_bufs, requests: Iterable[Tuple[int, np.ndarray, np.ndarray]]):
        """Copy every request's tokens [0, n_tokens) from the src pool into the dst pool, per head.
        Buffers are numpy uint8 arrays, one per (layer, plane, shard) in that order; dst is updated
        in place."""
        keep: list = []
        sp = self._pool(src_geom, src_bufs, keep)
        dp = self._pool(dst_geom, dst_bufs, keep)
        reqs = list(requests)
        n = len(reqs)
        ntok = np.asarray([int(r[0]) for r in reqs], np.int64)
        sids = [np.ascontiguousarray(r[1], np.int32) for r in reqs]
        dids = [np.ascontiguousarray(r[2], np.int32) for r in reqs]
        sp_arr = (ctypes.c_void_p * max(n, 1))(*[a.ctypes.data for a in sids])
        dp_arr = (ctypes.c_void_p * max(n, 1))(*[a.ctypes.data for a in dids])
        rc = self.lib.oracle_push(ctypes.byref(sp), ctypes.byref(dp), n, ntok.ctypes.data,
                                  ctypes.cast(sp_arr, _P), ctypes.cast(dp_arr, _P))
        if rc != 0:
            raise ValueError("oracle_push rejected its input (block id out of range or head mismatch)")

    # -- runs -----------------------------------------------------------------------------------
    def block_runs(self, src_ids, dst_ids):
        s = np.ascontiguousarray(src_ids, np.int32)
        d = np.ascontiguousarray(dst_ids, np.int32)
        n = len(s)
        rs, rd, rl = (np.zeros(max(n, 1), np.int32) for _ in range(3))
        nr = self.lib.oracle_block_runs(n, s.ctypes.data, d.ctypes.data, rs.ctypes.data, rd.ctypes.data,
                                        rl.ctypes.data)
        return rs[:nr].copy(), rd[:nr].copy(), rl[:nr].copy()

    def token_runs(self, n_tokens, bs_src, src_ids, bs_dst, dst_ids):
        s = np.ascontiguousarray(src_ids, np.int32)
        d = np.ascontiguousarray(dst_ids, np.int32)
        cap = max(int(n_tokens), 1)
        rs, rd, rl = (np.zeros(cap, np.int64) for _ in range(3))
        nr = self.lib.oracle_token_runs(int(n_tokens), bs_src, s.ctypes.data, bs_dst, d.ctypes.data,
                                        rs.ctypes.data, rd.ctypes.data, rl.ctypes.data)
        return rs[:nr].copy(), rd[:nr].copy(), rl[:nr].copy()

    # -- hashing --------------------------------------------------------------------------------
    def fnv1a64(self, data: bytes, h: int = None) -> int:
        buf = np.frombuffer(bytes(data), np.uint8) if len(data) else np.zeros(1, np.uint8)
        if h is None:
            h = int(self.lib.oracle_fnv64_offset_basis())
        return int(self.lib.oracle_fnv1a64(buf.ctypes.data, len(data), h))

    def offset_basis(self) -> int:
        return int(self.lib.oracle_fnv64_offset_basis())

    def block_hashes(self, tokens, block_size: int) -> np.ndarray:
        t = np.ascontiguousarray(tokens, np.uint32)
        out = np.zeros(max(len(t) // block_size, 1), np.uint64)
        n = self.lib.oracle_block_hashes(t.ctypes.data if len(t) else np.zeros(1, np.uint32).ctypes.data,
                                         len(t), block_size, out.ctypes.data)
        if n < 0:
            raise MemoryError("oracle_block_hashes")
        return out[:n].copy()

    # -- match ----------------------------------------------------------------------------------
    FILL_HOLES, KEEP_LAST = 1, 2

    def match(self, tokens, tok_off, block_size, local_keys, remote_hash, remote_blk, rem_off, threshold,
              free_blocks, flags=0, expiry=None, now=0):
        """Returns dict(local_hit, remote_hit, missing, push, dst_start, pair_src, pair_dst, status).
        flags: FILL_HOLES | KEEP_LAST; expiry (per session) with now: retention of the published span."""
        tokens = np.ascontiguousarray(tokens, np.uint32)
        tok_off = np.ascontiguousarray(tok_off, np.int64)
        n_s = len(tok_off) - 1
        keys = np.ascontiguousarray(local_keys, np.uint64)
        rh = np.ascontiguousarray(remote_hash, np.uint64)
        rb = np.ascontiguousarray(remote_blk, np.int32)
        ro = np.ascontiguousarray(rem_off, np.int64)
        fb = np.ascontiguousarray(free_blocks, np.int32)
        one = lambda a, dt: a if len(a) else np.zeros(1, dt)  # noqa: E731  (non-null pointers)
        tokens_, keys_, rh_, rb_, fb_ = one(tokens, np.uint32), one(keys, np.uint64), one(rh, np.uint64), \
            one(rb, np.int32), one(fb, np.int32)
        lh, rhit, miss, push = (np.zeros(max(n_s, 1), np.int32) for _ in range(4))
        dstart = np.zeros(max(n_s, 1), np.int64)
        cap = max(len(rb), 1)
        ps, pd = np.zeros(cap, np.int32), np.zeros(cap, np.int32)
        npairs = ctypes.c_int64(0)
        exp = None if expiry is None else np.ascontiguousarray(expiry, np.int64)
        rc = self.lib.oracle_match_ex(n_s, tokens_.ctypes.data, tok_off.ctypes.data, block_size,
                                      keys_.ctypes.data, len(keys), rh_.ctypes.data, rb_.ctypes.data,
                                      ro.ctypes.data, threshold, fb_.ctypes.data, len(fb), int(flags),
                                      None if exp is None else exp.ctypes.data, int(now),
                                      lh.ctypes.data, rhit.ctypes.data, miss.ctypes.data, push.ctypes.data,
                                      dstart.ctypes.data, ps.ctypes.data, pd.ctypes.data, ctypes.byref(npairs))
        if rc < 0:
            raise MemoryError("oracle_match")
        k = npairs.value
        return dict(local_hit=lh[:n_s].copy(), remote_hit=rhit[:n_s].copy(), missing=miss[:n_s].copy(),
                    push=push[:n_s].copy(), dst_start=dstart[:n_s].copy(), pair_src=ps[:k].copy(),
                    pair_dst=pd[:k].copy(), status=int(rc))


_default = None


def load() -> Oracle:
    """The oracle built from ``kvx_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
