"""Device-side helpers for the GPU parity tests: pools as slices of one torch allocation, seeded fills,
host copies for the oracle, and per-layer oracle checks."""
from __future__ import annotations

import numpy as np

import kvx_inputs
import oracle


def device_pool(geom, fill, seed=0, align=512):
    """One uint8 buffer per (layer, plane, shard), carved from one allocation. fill: 'bf16_normal',
    'fp8_bytes', or 'canary_<values kind>'."""
    import torch
    per = -(-geom.buffer_bytes // align) * align
    big = torch.empty(max(per * geom.n_buffers, align), dtype=torch.uint8, device="cuda")
    if fill == "bf16_normal":
        kvx_inputs.fill_bf16_normal(big, seed)
    elif fill == "fp8_bytes":
        kvx_inputs.fill_fp8_bytes(big, seed)
    elif fill.startswith("canary_"):
        kvx_inputs.fill_canary(big, fill[len("canary_"):])
    else:
        raise ValueError(fill)
    # the fill runs on the current stream; tests push from other streams, so it must be complete
    torch.cuda.synchronize()
    return [big[i * per:i * per + geom.buffer_bytes] for i in range(geom.n_buffers)], big


def layer_buffers(geom, bufs, layer):
    n = geom.n_planes * geom.n_shards
    return bufs[layer * n:(layer + 1) * n]


def host(bufs):
    return [b.cpu().numpy() for b in bufs]


def canary_host(geom, kind):
    """Host image of one canary-filled buffer."""
    if kind == "bf16_normal":
        return np.full(geom.buffer_bytes // 2, kvx_inputs.CANARY_BF16, np.uint16).view(np.uint8).copy()
    return np.full(geom.buffer_bytes, kvx_inputs.CANARY_FP8, np.uint8)


def check_layers(src_geom, src_bufs, dst_geom, dst_bufs, dst_before, requests, layers):
    """For each layer: the oracle's push of that layer on host copies, compared byte for byte with the
    device consumer buffers. dst_before(layer) gives that layer's consumer buffers before the push."""
    orc = oracle.load()
    sg1, dg1 = src_geom.replace(n_layers=1), dst_geom.replace(n_layers=1)
    for layer in layers:
        want = dst_before(layer)
        orc.push(sg1, host(layer_buffers(src_geom, src_bufs, layer)), dg1, want, requests)
        got = host(layer_buffers(dst_geom, dst_bufs, layer))
        for i, (a, b) in enumerate(zip(got, want)):
            if not np.array_equal(a, b):
                bad = np.flatnonzero(a != b)
                raise AssertionError(f"layer {layer} buffer {i}: {len(bad)} bytes differ, first at {bad[:8]}")
