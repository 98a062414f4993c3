"""Shared test helpers: host pools and two independent restatements of a push used to pin the oracle.

Neither restatement is the oracle's loop: ``numpy_route_push`` goes through numpy views (gather blocks,
reshape to tokens, concatenate head shards, split, scatter), ``dst_side_map`` starts from each
consumer byte and asks which producer byte must land there.
"""
from __future__ import annotations

import numpy as np

import kvx_inputs


def ceil_div(a, b):
    return -(-a // b)


def host_pool(geom, seed, fill="random"):
    """One uint8 numpy buffer per (layer, plane, shard)."""
    bufs = []
    for i in range(geom.n_buffers):
        if fill == "random":
            bufs.append(kvx_inputs.host_random_bytes(geom.buffer_bytes, seed * 1000 + i))
        else:
            bufs.append(np.full(geom.buffer_bytes, fill, np.uint8))
    return bufs


def nhd_view(geom, buf, hb):
    """A [block][slot][head][bytes] numpy view of one buffer, whatever its layout (writes go through)."""
    if getattr(geom, "layout", 0) == 1:
        return buf.reshape(geom.n_blocks, geom.heads_per_shard, geom.block_size, hb).transpose(0, 2, 1, 3)
    return buf.reshape(geom.n_blocks, geom.block_size, geom.heads_per_shard, hb)


def numpy_route_push(src_geom, src_bufs, dst_geom, dst_bufs, requests):
    """The push written with numpy tensor views; returns new dst buffers."""
    out = [b.copy() for b in dst_bufs]
    hb = src_geom.head_dim * src_geom.elem_bytes
    for (n, sids, dids) in requests:
        if n == 0:
            continue
        nbs, nbd = ceil_div(n, src_geom.block_size), ceil_div(n, dst_geom.block_size)
        for l in range(src_geom.n_layers):
            for p in range(src_geom.n_planes):
                shards = []
                for s in range(src_geom.n_shards):
                    v = nhd_view(src_geom, src_bufs[(l * src_geom.n_planes + p) * src_geom.n_shards + s], hb)
                    shards.append(v[np.asarray(sids[:nbs])].reshape(-1, src_geom.heads_per_shard, hb)[:n])
                tokens = np.concatenate(shards, axis=1)      # [n, all heads, head bytes]
                for d in range(dst_geom.n_shards):
                    part = tokens[:, d * dst_geom.heads_per_shard:(d + 1) * dst_geom.heads_per_shard]
                    v = nhd_view(dst_geom, out[(l * dst_geom.n_planes + p) * dst_geom.n_shards + d], hb)
                    idx = np.asarray(dids[:nbd])
                    cur = v[idx].reshape(-1, dst_geom.heads_per_shard, hb)
                    cur[:n] = part
                    v[idx] = cur.reshape(nbd, dst_geom.block_size, dst_geom.heads_per_shard, hb)
    return out


def dst_side_map(src_geom, src_bufs, dst_geom, dst_bufs, requests):
    """Per consumer byte: find the (request, token, head) that owns it and fetch the producer byte.
    Python loops; tiny inputs only. Returns new dst buffers."""
    out = [b.copy() for b in dst_bufs]
    hb = src_geom.head_dim * src_geom.elem_bytes
    owner = {}
    for r, (n, sids, dids) in enumerate(requests):
        for i in range(ceil_div(n, dst_geom.block_size)):
            owner[int(dids[i])] = (r, i)
    for l in range(dst_geom.n_layers):
        for p in range(dst_geom.n_planes):
            for d in range(dst_geom.n_shards):
                buf = out[(l * dst_geom.n_planes + p) * dst_geom.n_shards + d]
                for byte in range(dst_geom.buffer_bytes):
                    head_slot, within = divmod(byte, hb)
                    if getattr(dst_geom, "layout", 0) == 1:
                        blk_head, slot = divmod(head_slot, dst_geom.block_size)
                        blk, hd = divmod(blk_head, dst_geom.heads_per_shard)
                    else:
                        row, hd = divmod(head_slot, dst_geom.heads_per_shard)
                        blk, slot = divmod(row, dst_geom.block_size)
                    if blk not in owner:
                        continue
                    r, i = owner[blk]
                    n, sids, _ = requests[r]
                    t = i * dst_geom.block_size + slot
                    if t >= n:
                        continue
                    g = d * dst_geom.heads_per_shard + hd
                    s, hs = divmod(g, src_geom.heads_per_shard)
                    sblk, sslot = divmod(t, src_geom.block_size)
                    sb = int(sids[sblk])
                    if getattr(src_geom, "layout", 0) == 1:
                        sidx = (sb * src_geom.heads_per_shard + hs) * src_geom.block_size + sslot
                    else:
                        sidx = (sb * src_geom.block_size + sslot) * src_geom.heads_per_shard + hs
                    sbuf = src_bufs[(l * src_geom.n_planes + p) * src_geom.n_shards + s]
                    buf[byte] = sbuf[sidx * hb + within]
    return out


def random_requests(rng, src_geom, dst_geom, n_reqs, max_tokens):
    """Random request lengths and random (unique-per-side) block ids."""
    for _ in range(1000):   # redraw until both pools can hold every request
        lens = [int(x) for x in rng.integers(0, max_tokens + 1, n_reqs)]
        need_s = [ceil_div(n, src_geom.block_size) for n in lens]
        need_d = [ceil_div(n, dst_geom.block_size) for n in lens]
        if sum(need_s) <= src_geom.n_blocks and sum(need_d) <= dst_geom.n_blocks:
            break
    else:
        raise ValueError("pools too small for the requested lengths")
    sp = rng.permutation(src_geom.n_blocks).astype(np.int32)
    dp = rng.permutation(dst_geom.n_blocks).astype(np.int32)
    reqs, ps, pd = [], 0, 0
    for n, a, b in zip(lens, need_s, need_d):
        reqs.append((n, sp[ps:ps + a].copy(), dp[pd:pd + b].copy()))
        ps += a
        pd += b
    return reqs
