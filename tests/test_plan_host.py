"""Host-side tests of libkvx.so (no GPU): exported symbols, plan validation, merged runs against the
oracle, and the tile table replayed on the CPU with the copy kernel's semantics against the oracle.

kvx_plan makes no CUDA call, so the pools here carry fake, well-separated device addresses; the
replay uses numpy host buffers addressed by the tile offsets."""
import os
import re

import numpy as np
import pytest

import kvx_inputs
import oracle
from helpers import host_pool, random_requests

kvx = pytest.importorskip("disaggregated_prefill_decode_gb300.kvx")

PoolGeom = kvx_inputs.PoolGeom
HEADER = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", "include", "kvx.h")


def fake_pool(geom, base, align=256):
    stride = -(-geom.buffer_bytes // align) * align + align
    return kvx.Pool(geom, [base + i * stride for i in range(geom.n_buffers)])


def pools(sg, dg):
    return fake_pool(sg, 1 << 40), fake_pool(dg, 1 << 44)


def reqs_of(w):
    return [(r.n_tokens, r.src_ids, r.dst_ids) for r in w.requests]


def declared_functions():
    text = open(HEADER).read()
    return set(re.findall(r"^\s*(?:kvx_status|const char \*|int64_t)\s*(kvx_\w+)\s*\(", text, re.M))


def test_every_declared_symbol_is_exported():
    declared = declared_functions()
    assert {"kvx_plan", "kvx_push_layer", "kvx_sync", "kvx_match_prefix"} <= declared
    for name in sorted(declared):
        assert hasattr(kvx._lib, name), name
        assert name in kvx.EXPORTED, name


def test_status_strings_and_version():
    assert kvx.kvx_status_str(kvx.KVX_OK) == "KVX_OK"
    assert kvx.kvx_status_str(kvx.KVX_ETIMEDOUT) == "KVX_ETIMEDOUT"
    assert "sm_103a" in kvx.kvx_version()


def test_runs_match_oracle_on_workloads():
    orc = oracle.load()
    for make in (kvx_inputs.tiny, lambda: kvx_inputs.qwen3_32b_single(n_layers=1),
                 lambda: kvx_inputs.qwen3_32b_batched(n_layers=1),
                 lambda: kvx_inputs.tp4_to_tp1_remap(n_layers=1)):
        w = make()
        sp, dp = pools(w.src, w.dst)
        plan = kvx.kvx_plan(sp, dp, reqs_of(w))
        rs, rd, rl = kvx.kvx_plan_runs(plan)
        want = [orc.token_runs(r.n_tokens, w.src.block_size, r.src_ids, w.dst.block_size, r.dst_ids)
                for r in w.requests]
        assert np.array_equal(rs, np.concatenate([x[0] for x in want]))
        assert np.array_equal(rd, np.concatenate([x[1] for x in want]))
        assert np.array_equal(rl, np.concatenate([x[2] for x in want]))
        info = kvx.kvx_plan_get_info(plan)
        heads = w.src.n_shards * w.src.heads_per_shard
        assert info["bytes_per_layer"] == sum(r.n_tokens for r in w.requests) * heads * w.src.head_dim * \
            w.src.elem_bytes * w.src.n_planes
        assert info["strided"] == (w.name == "tp4_to_tp1_remap")
        kvx.kvx_plan_destroy(plan)


def replay_tiles(plan, sg, src, dg, dst):
    """The copy kernel's semantics on the CPU: each tile, for each (layer, plane)."""
    info = kvx.kvx_plan_get_info(plan)
    tiles = kvx.kvx_plan_tiles(plan)
    assert len(tiles) == info["n_tiles"]
    out = [b.copy() for b in dst]
    for l in range(sg.n_layers):
        for p in range(sg.n_planes):
            for t in tiles:
                sb = src[(l * sg.n_planes + p) * sg.n_shards + t["src_shard"]]
                db = out[(l * dg.n_planes + p) * dg.n_shards + t["dst_shard"]]
                so, do, n = int(t["src_off"]), int(t["dst_off"]), int(t["n"])
                if not info["strided"]:
                    assert n <= info["tile_bytes"] and n % info["vec_bytes"] == 0
                    db[do:do + n] = sb[so:so + n]
                else:
                    w, sp_, dp_ = info["width"], info["src_pitch"], info["dst_pitch"]
                    shp, dhp = info["src_head_pitch"], info["dst_head_pitch"]
                    assert n * max(int(t["heads"]), 1) * w <= max(info["tile_bytes"], w)
                    for h in range(max(int(t["heads"]), 1)):
                        for r in range(n):
                            s0, d0 = so + h * shp + r * sp_, do + h * dhp + r * dp_
                            db[d0:d0 + w] = sb[s0:s0 + w]
    return out


CASES = {
    "equal": (PoolGeom(2, 2, 1, 2, 4, 2, 4, 12), PoolGeom(2, 2, 1, 2, 4, 2, 4, 12)),
    "merge4to1_bs4to8": (PoolGeom(1, 2, 4, 1, 8, 2, 4, 10), PoolGeom(1, 2, 1, 4, 8, 2, 8, 6)),
    "split1to2_bs8to2": (PoolGeom(1, 1, 1, 4, 8, 2, 8, 5), PoolGeom(1, 1, 2, 2, 8, 2, 2, 20)),
    "merge2to1_equal_bs": (PoolGeom(1, 2, 2, 2, 16, 2, 4, 9), PoolGeom(1, 2, 1, 4, 16, 2, 4, 9)),
    "bs1": (PoolGeom(1, 2, 1, 2, 8, 1, 1, 24), PoolGeom(1, 2, 1, 2, 8, 1, 1, 24)),
    "odd_head_bytes": (PoolGeom(1, 1, 2, 1, 3, 1, 3, 9), PoolGeom(1, 1, 1, 2, 3, 1, 5, 7)),
    "mla576": (PoolGeom(2, 1, 1, 1, 576, 1, 4, 8), PoolGeom(2, 1, 1, 1, 576, 1, 4, 8)),
    "hnd_equal": (PoolGeom(1, 2, 2, 3, 8, 2, 4, 10, 1), PoolGeom(1, 2, 2, 3, 8, 2, 4, 10, 1)),
    "hnd_to_hnd_bs4to8": (PoolGeom(1, 1, 1, 4, 8, 2, 4, 12, 1), PoolGeom(1, 1, 1, 4, 8, 2, 8, 6, 1)),
    "nhd_to_hnd_merge": (PoolGeom(1, 2, 4, 1, 8, 2, 4, 10), PoolGeom(1, 2, 1, 4, 8, 2, 8, 6, 1)),
    "hnd_to_nhd_split": (PoolGeom(1, 1, 1, 4, 8, 2, 8, 5, 1), PoolGeom(1, 1, 2, 2, 8, 2, 2, 20)),
}


def test_head_major_plans_group_heads_per_tile():
    """A plan with a head-major side copies groups of heads per tile (the heads one producer shard and
    one consumer shard share, as many as fit tile_bytes), not one tile per head."""
    sg = PoolGeom(1, 2, 1, 8, 128, 2, 16, 64)
    dg = sg.replace(layout=1)
    sp, dp = pools(sg, dg)
    reqs = [(16 * 10, np.arange(10, dtype=np.int32), np.arange(20, 30, dtype=np.int32))]
    plan = kvx.kvx_plan_ex(sp, dp, reqs, {"tile_bytes": 16384})
    info = kvx.kvx_plan_get_info(plan)
    tiles = kvx.kvx_plan_tiles(plan)
    assert info["src_head_pitch"] == 256 and info["dst_head_pitch"] == 16 * 256
    assert len(tiles) == 10 * 2 and (tiles["heads"] == 4).all() and (tiles["n"] == 16).all()
    # head-group tiles move as tensor-map copies (4-stage ring) unless another kernel is asked for;
    # equal head-major layouts copy whole blocks and keep the bulk kernel
    assert (info["kernel"], info["threads"], info["bulk_stages"]) == (kvx.KVX_KERNEL_TENSOR, 32, 4)
    kvx.kvx_plan_destroy(plan)
    plan = kvx.kvx_plan_ex(sp, dp, reqs, {"kernel": kvx.KVX_KERNEL_STAGED})
    info = kvx.kvx_plan_get_info(plan)
    assert (info["kernel"], info["threads"]) == (kvx.KVX_KERNEL_STAGED, 128)
    assert info["tile_bytes"] == 4 * 16 * 256                  # other kernels: head groups of up to 16 KiB
    kvx.kvx_plan_destroy(plan)
    # the default tile of a TENSOR plan is a head group that divides the shared heads, up to 32 KiB
    # (here a whole block of 8 heads), in a 2-stage ring; asked-for TENSOR takes the same
    for opts in ({}, {"kernel": kvx.KVX_KERNEL_TENSOR}):
        plan = kvx.kvx_plan_ex(sp, dp, reqs, opts)
        tiles = kvx.kvx_plan_tiles(plan)
        info = kvx.kvx_plan_get_info(plan)
        assert (info["kernel"], info["tile_bytes"], info["bulk_stages"]) == (kvx.KVX_KERNEL_TENSOR, 8 * 16 * 256, 2)
        assert (tiles["heads"] == 8).all() and (tiles["n"] == 16).all()
        kvx.kvx_plan_destroy(plan)
    # head rows no tensor map can describe (24 bytes: not a multiple of 16) run the persistent kernel
    s24, d24 = sg.replace(head_dim=12), dg.replace(head_dim=12)
    p24, q24 = pools(s24, d24)
    plan = kvx.kvx_plan(p24, q24, reqs)
    assert (kvx.kvx_plan_get_info(plan)["kernel"], kvx.kvx_plan_get_info(plan)["threads"]) == (kvx.KVX_KERNEL_PERSIST, 128)
    kvx.kvx_plan_destroy(plan)
    plan = kvx.kvx_plan_ex(sp, dp, reqs, {"tile_bytes": 16384, "kernel": kvx.KVX_KERNEL_BULK})
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_BULK
    kvx.kvx_plan_destroy(plan)
    hp, hq = pools(dg, dg)
    plan = kvx.kvx_plan(hp, hq, reqs)
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_BULK
    kvx.kvx_plan_destroy(plan)
    # head-major -> token-major, and head-major pools of different block sizes: head groups again
    for a, b in ((dg, sg), (dg, dg.replace(block_size=32, n_blocks=32))):
        ap, bp = pools(a, b)
        nd = 16 * 10 // b.block_size
        rq = [(16 * 10, np.arange(10, dtype=np.int32), np.arange(10, 10 + nd, dtype=np.int32))]
        plan = kvx.kvx_plan(ap, bp, rq)
        i = kvx.kvx_plan_get_info(plan)
        assert (i["kernel"], i["threads"]) == (kvx.KVX_KERNEL_TENSOR, 32)
        kvx.kvx_plan_destroy(plan)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("tile_bytes", [16, 48, 1024, 16384])
def test_tile_replay_equals_oracle(name, tile_bytes):
    sg, dg = CASES[name]
    rng = np.random.default_rng(len(name) * 7 + tile_bytes)
    max_tok = min(sg.n_blocks * sg.block_size, dg.n_blocks * dg.block_size) // 3
    reqs = random_requests(rng, sg, dg, 3, max_tok)
    sp, dp = pools(sg, dg)
    plan = kvx.kvx_plan_ex(sp, dp, reqs, {"tile_bytes": tile_bytes})
    src = host_pool(sg, 5)
    dst = host_pool(dg, 0, fill=0x3C)
    got = replay_tiles(plan, sg, src, dg, dst)
    oracle.load().push(sg, src, dg, dst, reqs)
    for a, b in zip(got, dst):
        assert np.array_equal(a, b)
    kvx.kvx_plan_destroy(plan)


def test_tile_replay_tiny_workload():
    w = kvx_inputs.tiny()
    sp, dp = pools(w.src, w.dst)
    plan = kvx.kvx_plan(sp, dp, reqs_of(w))
    src = host_pool(w.src, 1)
    dst = host_pool(w.dst, 0, fill=0xAD)
    got = replay_tiles(plan, w.src, src, w.dst, dst)
    oracle.load().push(w.src, src, w.dst, dst, reqs_of(w))
    assert all(np.array_equal(a, b) for a, b in zip(got, dst))
    kvx.kvx_plan_destroy(plan)


def test_vector_width_follows_alignment():
    g = PoolGeom(1, 1, 1, 2, 64, 2, 16, 8)
    sp, dp = pools(g, g)
    pl = kvx.kvx_plan(sp, dp, [(20, [0, 1], [2, 3])])
    assert kvx.kvx_plan_get_info(pl)["vec_bytes"] == 16
    kvx.kvx_plan_destroy(pl)
    sp8 = kvx.Pool(g, [(1 << 40) + 8])
    pl = kvx.kvx_plan(sp8, dp, [(20, [0, 1], [2, 3])])
    assert kvx.kvx_plan_get_info(pl)["vec_bytes"] == 8
    kvx.kvx_plan_destroy(pl)
    g3 = PoolGeom(1, 1, 1, 1, 3, 1, 4, 8)
    sp, dp = pools(g3, g3)
    pl = kvx.kvx_plan(sp, dp, [(5, [0, 1], [2, 3])])
    assert kvx.kvx_plan_get_info(pl)["vec_bytes"] == 1
    kvx.kvx_plan_destroy(pl)


def test_empty_plans():
    g = PoolGeom(2, 2, 1, 2, 64, 2, 16, 8)
    sp, dp = pools(g, g)
    for reqs in ([], [(0, [], [])], [(0, [5], [6])]):
        pl = kvx.kvx_plan(sp, dp, reqs)
        info = kvx.kvx_plan_get_info(pl)
        assert info["n_runs"] == 0 and info["n_tiles"] == 0 and info["bytes_per_layer"] == 0
        assert kvx.kvx_sync(pl, 0) == kvx.KVX_OK                # nothing pushed: no device call
        assert kvx.kvx_plan_layer_states(pl).tolist() == [kvx.KVX_LAYER_IDLE] * 2
        kvx.kvx_plan_destroy(pl)


def expect(status, fn):
    with pytest.raises(kvx.KvxError) as ei:
        fn()
    assert ei.value.status == status, str(ei.value)
    assert kvx.kvx_last_error()


def test_validation_errors():
    g = PoolGeom(2, 2, 1, 2, 64, 2, 16, 8)
    sp, dp = pools(g, g)
    ok = (20, np.array([0, 1]), np.array([2, 3]))
    expect(kvx.KVX_ERANGE, lambda: kvx.kvx_plan(sp, dp, [(20, [0, 8], [2, 3])]))       # id == n_blocks
    expect(kvx.KVX_ERANGE, lambda: kvx.kvx_plan(sp, dp, [(20, [0, 1], [-1, 3])]))      # negative id
    expect(kvx.KVX_ERANGE, lambda: kvx.kvx_plan(sp, dp, [(40, [0, 1], [2, 3])]))       # too few ids
    expect(kvx.KVX_EOVERLAP, lambda: kvx.kvx_plan(sp, dp, [ok, (5, [4], [3])]))        # dst shared
    expect(kvx.KVX_EOVERLAP, lambda: kvx.kvx_plan(sp, dp, [(20, [0, 1], [5, 5])]))     # dst twice
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, dp, [(-1, [], [])]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, sp, [ok]))                         # same memory
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, kvx.Pool(g, dp.buffers[:3] + [dp.buffers[0]]), [ok]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, fake_pool(g.replace(n_layers=3), 1 << 44), [ok]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, fake_pool(g.replace(heads_per_shard=3), 1 << 44), [ok]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(sp, fake_pool(g.replace(head_dim=32, heads_per_shard=4), 1 << 44),
                                                [ok]))
    g6a, g6b = PoolGeom(1, 1, 3, 2, 8, 2, 4, 8), PoolGeom(1, 1, 2, 3, 8, 2, 4, 8)
    expect(kvx.KVX_EUNSUPPORTED, lambda: kvx.kvx_plan(fake_pool(g6a, 1 << 40), fake_pool(g6b, 1 << 44), [ok]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(fake_pool(g.replace(block_size=0), 1 << 40), dp, [ok]))
    expect(kvx.KVX_EUNSUPPORTED, lambda: kvx.kvx_plan(fake_pool(g.replace(layout=2), 1 << 40), dp, [ok]))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"tile_bytes": 24}))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"threads": 48}))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"layers_per_launch": -1}))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan(kvx.Pool(g, [0] * g.n_buffers), dp, [ok]))
    pl = kvx.kvx_plan(sp, dp, [ok])
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_inject_failure(pl, 2))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_push_layer(pl, 2))                # layer out of range, before CUDA
    kvx.kvx_plan_destroy(pl)


def test_requests_keep_extra_ids_unused():
    """ids past ceil(n_tokens / block_size) are ignored, so they may repeat."""
    g = PoolGeom(1, 1, 1, 1, 8, 2, 4, 8)
    sp, dp = pools(g, g)
    pl = kvx.kvx_plan(sp, dp, [(4, [0, 0, 0], [1, 1, 1]), (3, [2], [2])])
    assert kvx.kvx_plan_get_info(pl)["n_runs"] == 2
    kvx.kvx_plan_destroy(pl)


def test_timing_flag_validation():
    g = PoolGeom(1, 1, 1, 2, 64, 2, 16, 8)
    sp, dp = pools(g, g)
    ok = (20, [0, 1], [2, 3])
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"flags": 2}))
    plain = kvx.kvx_plan(sp, dp, [ok])
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_push_times(plain))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_push_times_ns(plain))
    kvx.kvx_plan_destroy(plain)
    timed = kvx.kvx_plan_ex(sp, dp, [ok], {"flags": kvx.KVX_PLAN_TIMING})
    s, e = kvx.kvx_plan_push_times(timed)
    assert len(s) == 0 and len(e) == 0                       # nothing synced yet
    kvx.kvx_plan_destroy(timed)


def test_kernel_resolution():
    g = PoolGeom(1, 2, 1, 8, 128, 2, 16, 8)
    sp, dp = pools(g, g)
    ok = (20, [0, 1], [2, 3])
    def kern(opts, a=sp, b=dp):
        p = kvx.kvx_plan_ex(a, b, [ok], opts)
        k = kvx.kvx_plan_get_info(p)["kernel"]
        kvx.kvx_plan_destroy(p)
        return k
    assert kern({}) == kvx.KVX_KERNEL_BULK
    assert kern({"tile_bytes": 65536}) == kvx.KVX_KERNEL_BULK                       # 3 x 64 KiB ring fits
    assert kern({"tile_bytes": 131072}) == kvx.KVX_KERNEL_PERSIST
    assert kern({"kernel": kvx.KVX_KERNEL_TILE}) == kvx.KVX_KERNEL_TILE
    assert kern({"kernel": kvx.KVX_KERNEL_BULK}) == kvx.KVX_KERNEL_BULK
    assert kern({"kernel": kvx.KVX_KERNEL_BULK, "tile_bytes": 131072}) == kvx.KVX_KERNEL_PERSIST  # ring too big
    assert kern({"kernel": kvx.KVX_KERNEL_TENSOR}) == kvx.KVX_KERNEL_BULK        # no head-major side: plain bulk
    assert kern({"kernel": kvx.KVX_KERNEL_STAGED}) == kvx.KVX_KERNEL_BULK        # contiguous tiles: plain bulk
    sp8 = kvx.Pool(g, [(1 << 40) + 8, (1 << 40) + 8 + (1 << 30)])
    assert kern({"kernel": kvx.KVX_KERNEL_BULK}, sp8, dp) == kvx.KVX_KERNEL_PERSIST                  # 8-byte aligned
    gs, gd = PoolGeom(1, 2, 2, 4, 128, 2, 16, 8), PoolGeom(1, 2, 1, 8, 128, 2, 16, 8)
    assert kern({}, fake_pool(gs, 1 << 40), fake_pool(gd, 1 << 44)) == kvx.KVX_KERNEL_BULK          # strided
    p = kvx.kvx_plan_ex(fake_pool(gs, 1 << 40), fake_pool(gd, 1 << 44), [ok], None)
    assert kvx.kvx_plan_get_info(p)["bulk_stages"] == 3                         # strided default ring
    kvx.kvx_plan_destroy(p)
    assert kern({"tile_bytes": 512}, fake_pool(gs, 1 << 40), fake_pool(gd, 1 << 44)) == \
        kvx.KVX_KERNEL_PERSIST                                                  # a 1024-byte row exceeds the stage
    gs8 = PoolGeom(1, 2, 2, 1, 4, 2, 16, 8)                                     # 8-byte rows: not 16-byte aligned
    gd8 = PoolGeom(1, 2, 1, 2, 4, 2, 16, 8)
    assert kern({"kernel": kvx.KVX_KERNEL_BULK}, fake_pool(gs8, 1 << 40), fake_pool(gd8, 1 << 44)) == \
        kvx.KVX_KERNEL_PERSIST
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"kernel": 9}))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"ctas_per_sm": 99}))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"lanes": 9}))
    p = kvx.kvx_plan(sp, dp, [ok])
    assert kvx.kvx_plan_get_info(p)["lanes"] in (1, 2, 3, 4)                  # by the process's hardware queues
    assert kvx.kvx_plan_get_info(p)["bulk_stages"] == 3
    kvx.kvx_plan_destroy(p)
    # AUTO by size: a layer push reading >= 128 MiB runs PERSIST with 128 threads unless asked otherwise
    gl = PoolGeom(1, 2, 1, 8, 128, 2, 16, 5000)
    big = (40000, list(range(2500)), list(range(2500)))                        # 40000 x 2 KiB x 2 planes
    def shape(opts):
        p = kvx.kvx_plan_ex(fake_pool(gl, 1 << 40), fake_pool(gl, 1 << 44), [big], opts)
        i = kvx.kvx_plan_get_info(p)
        kvx.kvx_plan_destroy(p)
        return i["kernel"], i["threads"], i["bytes_per_layer"]
    assert shape(None) == (kvx.KVX_KERNEL_PERSIST, 128, 40000 * 2048 * 2)
    assert shape({"threads": 512})[:2] == (kvx.KVX_KERNEL_PERSIST, 512)
    assert shape({"kernel": kvx.KVX_KERNEL_BULK})[:2] == (kvx.KVX_KERNEL_BULK, 32)
    assert shape({"kernel": kvx.KVX_KERNEL_PERSIST})[:2] == (kvx.KVX_KERNEL_PERSIST, 256)
    small = (32767 // 2, list(range(2500)), list(range(2500)))                 # just under 128 MiB
    p = kvx.kvx_plan_ex(fake_pool(gl, 1 << 40), fake_pool(gl, 1 << 44), [small], None)
    assert kvx.kvx_plan_get_info(p)["kernel"] == kvx.KVX_KERNEL_BULK
    kvx.kvx_plan_destroy(p)
    # ring stages: only instantiated counts; a ring over 192 KiB leaves the bulk kernel
    for bad in (1, 5, 7, 9, -1):
        expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_ex(sp, dp, [ok], {"bulk_stages": bad}))
    assert kern({"bulk_stages": 8, "tile_bytes": 24576}) == kvx.KVX_KERNEL_BULK             # 192 KiB
    assert kern({"bulk_stages": 8, "tile_bytes": 24592}) == kvx.KVX_KERNEL_PERSIST          # just over
    assert kern({"bulk_stages": 2, "tile_bytes": 49152}) == kvx.KVX_KERNEL_BULK
    p = kvx.kvx_plan_ex(sp, dp, [ok], {"bulk_stages": 6})
    assert kvx.kvx_plan_get_info(p)["bulk_stages"] == 6
    kvx.kvx_plan_set_opts(p, {"bulk_stages": 3})
    assert kvx.kvx_plan_get_info(p)["bulk_stages"] == 3
    kvx.kvx_plan_set_opts(p, {"kernel": kvx.KVX_KERNEL_PERSIST})
    assert kvx.kvx_plan_get_info(p)["bulk_stages"] == 0                                     # not a bulk plan
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_set_opts(p, {"bulk_stages": 5}))
    kvx.kvx_plan_destroy(p)


def test_head_group_default_tiles_divide_the_shared_heads():
    """Plans that map one head layout onto another cut each block segment into equal head groups: the
    largest divisor of the heads a producer shard and a consumer shard share that fits 32 KiB on the
    tensor-map kernel, so every group is one tensor-map box (6 shared heads of 256 B over 12-token
    blocks: all 6 in a tile; a TP1 -> TP2 split with 4 shared heads: 4; 8 heads of 512 B: 4)."""
    cases = [
        (PoolGeom(1, 2, 1, 6, 128, 2, 12, 40), PoolGeom(1, 2, 1, 6, 128, 2, 12, 40, 1), 6, 12),
        (PoolGeom(1, 2, 1, 8, 128, 2, 16, 40), PoolGeom(1, 2, 2, 4, 128, 2, 16, 40, 1), 4, 16),
        (PoolGeom(1, 2, 1, 8, 128, 2, 16, 40, 1), PoolGeom(1, 2, 1, 8, 128, 2, 32, 20), 8, 16),
        (PoolGeom(1, 2, 1, 8, 256, 2, 16, 40, 1), PoolGeom(1, 2, 1, 8, 256, 2, 16, 40), 4, 16),
    ]
    for sg, dg, k, n in cases:
        sp, dp = pools(sg, dg)
        n_tok = 4 * max(sg.block_size, dg.block_size)
        reqs = [(n_tok, np.arange(n_tok // sg.block_size, dtype=np.int32),
                 np.arange(3, 3 + n_tok // dg.block_size, dtype=np.int32))]
        plan = kvx.kvx_plan(sp, dp, reqs)
        info = kvx.kvx_plan_get_info(plan)
        tiles = kvx.kvx_plan_tiles(plan)
        assert info["kernel"] == kvx.KVX_KERNEL_TENSOR
        assert info["tile_bytes"] == k * n * sg.head_dim * sg.elem_bytes
        assert (np.maximum(tiles["heads"], 1) == k).all() and (tiles["n"] == n).all()
        total_heads = sg.n_shards * sg.heads_per_shard
        assert len(tiles) == (n_tok // n) * (total_heads // k)
        kvx.kvx_plan_destroy(plan)


def test_stall_hook_argument_checks():
    """kvx_plan_inject_stall needs a ring kernel and a layer of the plan; no CUDA call is made."""
    g = PoolGeom(2, 2, 1, 8, 128, 2, 16, 40)
    sp, dp = pools(g, g)
    reqs = [(64, np.arange(4, dtype=np.int32), np.arange(10, 14, dtype=np.int32))]
    for kernel, ok in ((kvx.KVX_KERNEL_BULK, True), (kvx.KVX_KERNEL_PERSIST, False), (kvx.KVX_KERNEL_TILE, False)):
        plan = kvx.kvx_plan_ex(sp, dp, reqs, {"kernel": kernel})
        if ok:
            kvx.kvx_plan_inject_stall(plan, 1)
        else:
            expect(kvx.KVX_EUNSUPPORTED, lambda: kvx.kvx_plan_inject_stall(plan, 1))
        kvx.kvx_plan_destroy(plan)
    plan = kvx.kvx_plan(sp, dp, reqs)
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_inject_stall(plan, 2))
    expect(kvx.KVX_EINVAL, lambda: kvx.kvx_plan_inject_stall(plan, -1))
    kvx.kvx_plan_destroy(plan)
    hg, hd = PoolGeom(1, 2, 1, 8, 128, 2, 16, 40), PoolGeom(1, 2, 1, 8, 128, 2, 16, 40, 1)
    hp, hq = pools(hg, hd)
    for kernel in (kvx.KVX_KERNEL_TENSOR, kvx.KVX_KERNEL_STAGED):
        plan = kvx.kvx_plan_ex(hp, hq, reqs, {"kernel": kernel})
        kvx.kvx_plan_inject_stall(plan, 0)
        kvx.kvx_plan_destroy(plan)


_LANES_PROBE = """
import numpy as np
from kvx_inputs import PoolGeom
from disaggregated_prefill_decode_gb300 import kvx
g = PoolGeom(2, 2, 1, 8, 128, 2, 16, 40)
def pool(base):
    return kvx.Pool(g, [base + i * (g.buffer_bytes + 256) for i in range(g.n_buffers)])
reqs = [(64, np.arange(4, dtype=np.int32), np.arange(10, 14, dtype=np.int32))]
p = kvx.kvx_plan(pool(1 << 40), pool(1 << 44), reqs)
print(kvx.kvx_plan_get_info(p)["lanes"])
kvx.kvx_plan_set_opts(p, {"lanes": 0})
print(kvx.kvx_plan_get_info(p)["lanes"])
"""


@pytest.mark.parametrize("queues,lanes", [(None, 4), ("1", 1), ("2", 1), ("4", 2), ("6", 3), ("8", 4), ("32", 4),
                                          ("", 4), ("many", 4), ("0", 4)])
def test_default_lanes_follow_the_hardware_queues(queues, lanes):
    """The default lane count follows CUDA_DEVICE_MAX_CONNECTIONS as the process started: 4 lanes, or
    half the queues when that is fewer, at least 1 (8 queues, the runtime's default: 4)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k != "CUDA_DEVICE_MAX_CONNECTIONS"}
    if queues is not None:
        env["CUDA_DEVICE_MAX_CONNECTIONS"] = queues
    env["PYTHONPATH"] = os.pathsep.join([root, os.path.join(root, "tests"), env.get("PYTHONPATH", "")])
    out = subprocess.run([sys.executable, "-c", _LANES_PROBE], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(lanes), str(lanes)]
