"""GPU parity of the layer push through the C-ABI: the kvx copy on device against the oracle, byte for
byte (this is pure data movement: bit-exact is the only bar).

Small cases run every layer through the oracle; the full-size workloads (Qwen3-32B-shaped, 64 layers)
run in the launch configuration the benchmark times (one push per layer on a high-priority side
stream, gated on an event after the prefill fixture) and check sampled layers whole."""
import zlib

import numpy as np
import pytest

import kvx_inputs
import prefill_fixture
import oracle
from gpu_helpers import canary_host, check_layers, device_pool, host, layer_buffers

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


def reqs_of(w):
    return [(r.n_tokens, r.src_ids, r.dst_ids) for r in w.requests]


def push_all_layers(plan, n_layers, fixture_iters=2000, per_layer=True):
    """The benchmark's launch pattern: fixture on the main stream, event, push on a side stream."""
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=-1)
    if per_layer:
        for layer in range(n_layers):
            prefill_fixture.prefill(8, fixture_iters, stream=main)
            ev = torch.cuda.Event()
            ev.record(main)
            kvx.kvx_push_layer(plan, layer, side, ev)
    else:
        ev = torch.cuda.Event()
        ev.record(main)
        kvx.kvx_push_layers(plan, 0, n_layers, side, ev)
    return kvx.kvx_sync(plan, -1)


def run_workload(w, layers_to_check, opts=None, per_layer=True):
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w), opts)
    assert push_all_layers(plan, w.src.n_layers, per_layer=per_layer) == kvx.KVX_OK
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE] * w.src.n_layers
    per = w.dst.n_planes * w.dst.n_shards
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(per)],
                 reqs_of(w), layers_to_check)
    info = kvx.kvx_plan_get_info(plan)
    kvx.kvx_plan_destroy(plan)
    return info


def test_tiny_all_layers():
    w = kvx_inputs.tiny()
    run_workload(w, range(w.src.n_layers))


KERNELS = {"tile": 1, "persist": 2, "bulk": 3, "tensor": 4, "staged": 5}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("make", [
    lambda: kvx_inputs.qwen3_32b_single(n_layers=2),
    lambda: kvx_inputs.qwen3_32b_batched(n_layers=2, n_requests=6),
    lambda: kvx_inputs.tp4_to_tp1_remap(n_layers=2, n_requests=3),
], ids=["qwen3_32b_single", "qwen3_32b_batched", "tp4_to_tp1_remap"])
def test_reduced_workloads_all_layers(make, kernel):
    w = make()
    info = run_workload(w, range(w.src.n_layers), opts={"kernel": KERNELS[kernel]})
    assert info["vec_bytes"] == 16
    # strided plans run the bulk kernel too; TENSOR asked for on a plan with no head-major side is BULK,
    # and so is STAGED on a contiguous plan
    want = KERNELS[kernel]
    if kernel == "tensor" or (kernel == "staged" and not info["strided"]):
        want = kvx.KVX_KERNEL_BULK
    assert info["kernel"] == want


@pytest.mark.parametrize("lanes", [1, 2, 5])
def test_lanes(lanes):
    w = kvx_inputs.qwen3_32b_batched(n_layers=6, n_requests=4, len_range=(500, 3000))
    info = run_workload(w, range(6), opts={"lanes": lanes})
    assert info["lanes"] == lanes


@pytest.mark.parametrize("stages,tile_bytes", [(2, 49152), (3, 16384), (6, 8192), (8, 24576), (8, 4096)])
def test_bulk_ring_stages(stages, tile_bytes):
    w = kvx_inputs.qwen3_32b_batched(n_layers=2, n_requests=4, len_range=(100, 2000))
    info = run_workload(w, range(2), opts={"kernel": kvx.KVX_KERNEL_BULK, "tile_bytes": tile_bytes,
                                           "bulk_stages": stages})
    assert (info["kernel"], info["bulk_stages"]) == (kvx.KVX_KERNEL_BULK, stages)
    run_workload(w, range(2), opts={"kernel": kvx.KVX_KERNEL_BULK, "tile_bytes": tile_bytes, "bulk_stages": stages},
                 per_layer=False)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("tile_bytes,ctas", [(4096, 0), (16384, 2), (49152, 1)])
def test_kernels_launch_shapes(kernel, tile_bytes, ctas):
    w = kvx_inputs.qwen3_32b_batched(n_layers=2, n_requests=4, len_range=(100, 2000))
    run_workload(w, range(2), opts={"kernel": KERNELS[kernel], "tile_bytes": tile_bytes, "ctas_per_sm": ctas})
    run_workload(w, range(2), opts={"kernel": KERNELS[kernel], "tile_bytes": tile_bytes}, per_layer=False)


@pytest.mark.parametrize("name", ["qwen3_32b_single", "qwen3_32b_batched", "tp4_to_tp1_remap"])
def test_full_size_sampled_layers(name):
    """Full 64-layer workload in the benchmark's launch pattern; layers 0, 31, 63 checked whole."""
    w = kvx_inputs.PUSH_WORKLOADS[name]()
    run_workload(w, [0, 31, 63])


def test_all_layers_in_one_launch():
    w = kvx_inputs.qwen3_32b_batched(n_layers=3, n_requests=4)
    run_workload(w, range(3), per_layer=False)


@pytest.mark.parametrize("opts,launches", [({"layers_per_launch": 3}, [(0, 3), (3, 6), (6, 7)]),
                                           ({}, [(0, 4), (4, 7)]),                 # 64 MiB a layer: 4 a launch
                                           ({"lanes": 1}, [(0, 7)]),
                                           ({"lanes": 1, "layers_per_launch": 2}, [(0, 2), (2, 4), (4, 6), (6, 7)])])
def test_push_layers_split_into_launches(opts, launches):
    """kvx_push_layers over 7 layers in launches of layers_per_launch layers (by default about
    256 MiB moved per launch when lanes > 1): every layer lands, one timing entry per launch."""
    w = kvx_inputs.qwen3_32b_single(n_layers=7)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w),
                           dict(opts, flags=kvx.KVX_PLAN_TIMING))
    n0 = kvx.kvx_launch_count()
    assert push_all_layers(plan, 7, per_layer=False) == kvx.KVX_OK
    assert kvx.kvx_launch_count() - n0 == len(launches)
    assert len(kvx.kvx_plan_push_times_ns(plan)[0]) == len(launches)
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE] * 7
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(7))
    kvx.kvx_plan_destroy(plan)


def test_head_major_pool_in_pinned_host_memory():
    """A head-major consumer pool in pinned host memory, fed from a token-major device pool: head-group
    tiles written over the chip-to-chip link with plain stores, byte for byte against the oracle."""
    w = kvx_inputs.qwen3_32b_batched_nhd_to_hnd(n_layers=2)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    dst = [b.cpu().pin_memory() for b in dst]
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_PERSIST
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(2))
    kvx.kvx_plan_destroy(plan)


@pytest.mark.parametrize("side", ["src", "dst"])
@pytest.mark.parametrize("kernel", ["auto", "bulk"])
def test_pool_in_pinned_host_memory(side, kernel):
    """One pool in pinned host memory, reached over the chip-to-chip link: the plan's pushes copy it
    with plain loads and stores (the bulk copy path is kept to device memory, even when asked for),
    byte for byte against the oracle."""
    w = kvx_inputs.qwen3_32b_single(n_layers=2)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    if side == "src":
        src = [b.cpu().pin_memory() for b in src]
    else:
        dst = [b.cpu().pin_memory() for b in dst]
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w),
                           {"kernel": KERNELS[kernel] if kernel != "auto" else 0})
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_PERSIST
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(2))
    kvx.kvx_plan_destroy(plan)


def test_push_layers_notify_follows_every_launch():
    """The notification of a multi-layer push split over lanes is recorded after all its launches: a
    consumer stream that waits on it reads every layer complete."""
    w = kvx_inputs.qwen3_32b_single(n_layers=7)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w), {"layers_per_launch": 1})
    side, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    done = torch.cuda.Event()
    kvx.kvx_push_layer_notify(plan, 0, 7, side, None, done)
    consumer.wait_event(done)
    with torch.cuda.stream(consumer):
        copies = [[b.clone() for b in layer_buffers(w.dst, dst, layer)] for layer in range(7)]
    consumer.synchronize()
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    for layer in range(7):
        for a, b in zip(copies[layer], layer_buffers(w.dst, dst, layer)):
            assert torch.equal(a, b)
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(7))
    kvx.kvx_plan_destroy(plan)


@pytest.mark.parametrize("tile_bytes,threads", [(16, 32), (4096, 128), (16384, 256), (65536, 1024), (2064, 96)])
def test_launch_shapes(tile_bytes, threads):
    w = kvx_inputs.qwen3_32b_batched(n_layers=1, n_requests=3, len_range=(100, 900))
    run_workload(w, [0], opts={"tile_bytes": tile_bytes, "threads": threads})


GEOMS = {
    # name: (src, dst) -- block sizes 1/16/64, odd head bytes (narrow vectors), merges and splits
    "bs1": (PoolGeom(2, 2, 1, 2, 64, 2, 1, 300), PoolGeom(2, 2, 1, 2, 64, 2, 1, 300)),
    "bs64_to_16": (PoolGeom(2, 2, 1, 8, 128, 2, 64, 20), PoolGeom(2, 2, 1, 8, 128, 2, 16, 80)),
    "head_bytes_6": (PoolGeom(1, 2, 1, 3, 3, 2, 16, 40), PoolGeom(1, 2, 1, 3, 3, 2, 16, 40)),
    "head_bytes_3_merge": (PoolGeom(1, 1, 2, 1, 3, 1, 4, 50), PoolGeom(1, 1, 1, 2, 3, 1, 8, 25)),
    "head_bytes_12_split": (PoolGeom(1, 1, 1, 4, 6, 2, 8, 30), PoolGeom(1, 1, 4, 1, 6, 2, 4, 60)),
    "split1to2": (PoolGeom(2, 2, 1, 8, 128, 2, 16, 40), PoolGeom(2, 2, 2, 4, 128, 2, 16, 40)),
    "merge8to2": (PoolGeom(1, 2, 8, 1, 64, 2, 16, 40), PoolGeom(1, 2, 2, 4, 64, 2, 32, 20)),
    "mla576_fp8": (PoolGeom(2, 1, 1, 1, 576, 1, 64, 30), PoolGeom(2, 1, 1, 1, 576, 1, 64, 30)),
    "hnd_qwen_equal": (PoolGeom(2, 2, 1, 8, 128, 2, 16, 60, 1), PoolGeom(2, 2, 1, 8, 128, 2, 16, 60, 1)),
    "hnd_tp4_to_nhd_tp1_bs64": (PoolGeom(1, 2, 4, 2, 128, 2, 16, 60, 1), PoolGeom(1, 2, 1, 8, 128, 2, 64, 15)),
    "nhd_to_hnd_bs16to32": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 60), PoolGeom(1, 2, 1, 8, 128, 2, 32, 30, 1)),
    "hnd_odd_heads": (PoolGeom(1, 1, 1, 3, 3, 2, 8, 40, 1), PoolGeom(1, 1, 3, 1, 3, 2, 4, 80, 1)),
    "nhd_tp1_to_hnd_tp2": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 60), PoolGeom(1, 2, 2, 4, 128, 2, 16, 60, 1)),
    # tensor-map boxes: heads and block sizes that are not powers of two (box of 3 heads x 12 slots),
    # a head-major split with a block-size change, head rows of 16 and 2048 bytes
    "nhd_to_hnd_nonpow2": (PoolGeom(1, 2, 1, 6, 128, 2, 12, 50), PoolGeom(1, 2, 1, 6, 128, 2, 12, 50, 1)),
    "hnd_tp1_to_hnd_tp2_bs32": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 60, 1), PoolGeom(1, 2, 2, 4, 128, 2, 32, 30, 1)),
    "hnd_to_nhd_16byte_heads": (PoolGeom(2, 1, 1, 4, 8, 2, 16, 40, 1), PoolGeom(2, 1, 1, 4, 8, 2, 16, 40)),
    "nhd_to_hnd_2kib_heads": (PoolGeom(1, 1, 2, 2, 1024, 2, 8, 30), PoolGeom(1, 1, 1, 4, 1024, 2, 8, 30, 1)),
}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", sorted(GEOMS))
def test_geometry_sweep(name, kernel):
    from helpers import random_requests
    sg, dg = GEOMS[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    reqs = random_requests(rng, sg, dg, 4, min(sg.n_blocks * sg.block_size, dg.n_blocks * dg.block_size) // 4)
    kind = "fp8_bytes" if sg.elem_bytes == 1 else "bf16_normal"
    src, _ = device_pool(sg, kind, seed=7)
    dst, _ = device_pool(dg, "canary_" + kind)
    plan = kvx.kvx_plan_ex(kvx.Pool(sg, src), kvx.Pool(dg, dst), reqs, {"kernel": KERNELS[kernel]})
    assert push_all_layers(plan, sg.n_layers) == kvx.KVX_OK
    per = dg.n_planes * dg.n_shards
    check_layers(sg, src, dg, dst, lambda l: [canary_host(dg, kind) for _ in range(per)], reqs, range(sg.n_layers))
    kvx.kvx_plan_destroy(plan)


# Tensor-map plans: the box (box_n slots x box_k heads) is laid out in shared memory in the consumer's
# layout when a box is one contiguous span of the consumer (token-major: all of a shard's heads;
# head-major: all of a block's slots), else in the producer's when it is one of the producer's, else
# token-major; a side whose layout that is and which holds the box contiguously moves it by a plain bulk
# copy, the other through its tensor map. (name: src, dst, tile_bytes, the case it takes)
BOX_CASES = {
    "nhd_to_hnd_store_plain": (PoolGeom(2, 2, 1, 8, 128, 2, 16, 40), PoolGeom(2, 2, 1, 8, 128, 2, 16, 40, 1), 0),
    "hnd_to_nhd_store_plain": (PoolGeom(2, 2, 1, 8, 128, 2, 16, 40, 1), PoolGeom(2, 2, 1, 8, 128, 2, 16, 40), 0),
    "hnd_to_nhd_load_plain": (PoolGeom(2, 2, 1, 8, 128, 2, 16, 40, 1), PoolGeom(2, 2, 1, 8, 128, 2, 16, 40), 16384),
    "nhd_to_hnd_bs32_load_plain": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 60), PoolGeom(1, 2, 1, 8, 128, 2, 32, 30, 1), 0),
    "nhd_to_hnd_bs32_both_maps": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 60), PoolGeom(1, 2, 1, 8, 128, 2, 32, 30, 1), 16384),
    "hnd_tp1_to_hnd_tp2_both_plain": (PoolGeom(1, 2, 1, 8, 128, 2, 16, 40, 1), PoolGeom(1, 2, 2, 4, 128, 2, 16, 40, 1), 0),
    "nhd_to_hnd_6heads_store_plain": (PoolGeom(1, 2, 1, 6, 128, 2, 12, 50), PoolGeom(1, 2, 1, 6, 128, 2, 12, 50, 1), 0),
}


@pytest.mark.parametrize("name", sorted(BOX_CASES))
def test_tensor_box_orders(name):
    from helpers import random_requests
    sg, dg, tile_bytes = BOX_CASES[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    reqs = random_requests(rng, sg, dg, 4, min(sg.n_blocks * sg.block_size, dg.n_blocks * dg.block_size) // 4)
    src, _ = device_pool(sg, "bf16_normal", seed=11)
    dst, _ = device_pool(dg, "canary_bf16_normal")
    plan = kvx.kvx_plan_ex(kvx.Pool(sg, src), kvx.Pool(dg, dst), reqs, {"tile_bytes": tile_bytes})
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_TENSOR
    assert push_all_layers(plan, sg.n_layers) == kvx.KVX_OK
    per = dg.n_planes * dg.n_shards
    check_layers(sg, src, dg, dst, lambda l: [canary_host(dg, "bf16_normal") for _ in range(per)], reqs,
                 range(sg.n_layers))
    kvx.kvx_plan_destroy(plan)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_offsets_past_4gib(kernel):
    """One 4.9 GB buffer per side (150,000 blocks of 32 KiB): runs that start and end beyond 2^32 bytes,
    one that straddles it and one near the start; every copied block equals its source block and the
    blocks around them keep their canary."""
    g = PoolGeom(1, 1, 1, 8, 128, 2, 16, 150_000)
    bb = 16 * g.row_bytes
    src, _ = device_pool(g, "bf16_normal", seed=9)
    dst, _ = device_pool(g, "canary_bf16_normal")
    assert g.buffer_bytes > (1 << 32) + 8 * bb
    edge = (1 << 32) // bb                                             # first block past 4 GiB: 131072
    runs = [(edge - 3, edge + 1000, 7), (edge + 5000, edge - 2, 6), (10, 149_990, 4), (149_000, 20, 9)]
    reqs = [(n * 16, np.arange(sb, sb + n), np.arange(db, db + n)) for sb, db, n in runs]
    plan = kvx.kvx_plan_ex(kvx.Pool(g, src), kvx.Pool(g, dst), reqs, {"kernel": KERNELS[kernel]})
    assert push_all_layers(plan, 1) == kvx.KVX_OK
    kvx.kvx_plan_destroy(plan)
    canary = torch.tensor(kvx_inputs.CANARY_BF16 - 0x10000, dtype=torch.int16, device="cuda")
    s, d = src[0], dst[0]
    for sb, db, n in runs:
        assert torch.equal(d[db * bb:(db + n) * bb], s[sb * bb:(sb + n) * bb]), (sb, db, n)
        for nb in (db - 1, db + n):                                    # the neighbours keep the canary
            assert bool((d[nb * bb:(nb + 1) * bb].view(torch.int16) == canary).all()), nb


def test_one_huge_run_equals_one_copy():
    g = PoolGeom(2, 2, 1, 8, 128, 2, 16, 1100)
    src, _ = device_pool(g, "bf16_normal", seed=3)
    dst, _ = device_pool(g, "canary_bf16_normal")
    n_blk, off = 1000, 50
    plan = kvx.kvx_plan(kvx.Pool(g, src), kvx.Pool(g, dst), [(n_blk * 16, np.arange(n_blk), np.arange(off, off + n_blk))])
    assert kvx.kvx_plan_get_info(plan)["n_runs"] == 1
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    bb = 16 * g.row_bytes
    canary = torch.tensor(kvx_inputs.CANARY_BF16 - 0x10000, dtype=torch.int16, device="cuda")
    for s, d in zip(src, dst):
        assert torch.equal(d[off * bb:(off + n_blk) * bb], s[:n_blk * bb])
        assert bool((d[:off * bb].view(torch.int16) == canary).all())
        assert bool((d[(off + n_blk) * bb:].view(torch.int16) == canary).all())
    kvx.kvx_plan_destroy(plan)


def test_empty_plan_pushes_nothing():
    g = PoolGeom(2, 2, 1, 2, 64, 2, 16, 8)
    src, _ = device_pool(g, "bf16_normal", seed=1)
    dst, big = device_pool(g, "canary_bf16_normal")
    before = big.clone()
    plan = kvx.kvx_plan(kvx.Pool(g, src), kvx.Pool(g, dst), [(0, [], [])])
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    assert torch.equal(big, before)
    kvx.kvx_plan_destroy(plan)


def test_producer_unchanged_and_plan_reusable():
    w = kvx_inputs.qwen3_32b_batched(n_layers=2, n_requests=3)
    src, sbig = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    s_before = sbig.clone()
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    for _ in range(3):                                  # the same plan pushed three times
        assert push_all_layers(plan, 2) == kvx.KVX_OK
    assert torch.equal(sbig, s_before)
    per = w.dst.n_planes
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(per)],
                 reqs_of(w), range(2))
    kvx.kvx_plan_destroy(plan)


def test_push_ordered_after_prefill_rewrite():
    """The fixture rewrites each layer's producer KV just before its event; a push that started early
    would copy the stale bytes. The final consumer must equal the oracle on the final producer."""
    w = kvx_inputs.qwen3_32b_single(n_layers=4)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=-1)
    for layer in range(4):
        for b in layer_buffers(w.src, src, layer):
            prefill_fixture.prefill(16, 20000, b, b.numel(), seed=1000 + layer, stream=main)
        ev = torch.cuda.Event()
        ev.record(main)
        kvx.kvx_push_layer(plan, layer, side, ev)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(4))
    kvx.kvx_plan_destroy(plan)


def test_push_ordered_after_graph_replayed_prefill():
    """The prefill captured once into a CUDA graph (each layer's ready event an external event-record
    node) and replayed per step, the push of every layer gated on its event. Before each replay the
    producer is zeroed and the consumer re-filled with canaries on the main stream, so a push that ran
    ahead of the replay's rewrite would leave zeros behind; the consumer must equal the oracle."""
    w = kvx_inputs.qwen3_32b_single(n_layers=3)
    src, src_big = device_pool(w.src, w.values, seed=w.seed)
    dst, dst_big = device_pool(w.dst, "canary_" + w.values)
    cap = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(3)]
    for ev in ready:
        ev.record()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for layer in range(3):
            for b in layer_buffers(w.src, src, layer):
                prefill_fixture.prefill(16, 20000, b, b.numel(), seed=500 + layer, stream=cap)
            prefill_fixture.prefill(1, 1, stream=cap, done=ready[layer])
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=-1)
    for rep in range(3):
        src_big.zero_()
        kvx_inputs.fill_canary(dst_big, w.values)
        g.replay()
        plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
        for layer in range(3):
            kvx.kvx_push_layer(plan, layer, side, ready[layer])
        assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
        kvx.kvx_plan_destroy(plan)
        main.synchronize()
        assert not all(bool((b == 0).all()) for b in layer_buffers(w.src, src, 2))   # the replay rewrote it
        check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)],
                     reqs_of(w), range(3))


def test_sync_timeout_then_completion():
    """A long (bounded) fixture holds the stream; a 1 ms deadline times out, a later sync completes."""
    w = kvx_inputs.tiny()
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    side = torch.cuda.Stream()
    prefill_fixture.prefill(1, 30_000_000, stream=side)          # ~tens of ms of dependent integer work
    kvx.kvx_push_layer(plan, 0, side)
    kvx.kvx_push_layer(plan, 1, side)
    assert kvx.kvx_sync(plan, 1000) == kvx.KVX_ETIMEDOUT
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_PENDING] * 2
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(2))
    kvx.kvx_plan_destroy(plan)


def test_injected_failure_reports_failed_layer():
    w = kvx_inputs.tiny()
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    kvx.kvx_plan_inject_failure(plan, 1)
    assert push_all_layers(plan, 2) == kvx.KVX_EFAILED
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE, kvx.KVX_LAYER_FAILED]
    assert push_all_layers(plan, 2) == kvx.KVX_OK                # the injection fires once
    assert kvx.kvx_plan_layer_states(plan).tolist() == [kvx.KVX_LAYER_DONE] * 2
    kvx.kvx_plan_destroy(plan)


def test_launch_count_grows():
    n0, f0 = kvx.kvx_launch_count(), prefill_fixture.launch_count()
    test_tiny_all_layers()
    assert kvx.kvx_launch_count() >= n0 + 2                     # 2 pushes
    assert prefill_fixture.launch_count() == f0 + 2             # 2 fixtures, counted by their own library


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_push_times_of_timing_plan(kernel):
    """Timing plans: the copy kernels stamp the GPU's global timer (first CTA start, last CTA end)."""
    w = kvx_inputs.qwen3_32b_single(n_layers=4)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w),
                           {"flags": kvx.KVX_PLAN_TIMING, "kernel": KERNELS[kernel]})
    assert push_all_layers(plan, 4) == kvx.KVX_OK
    s, e = kvx.kvx_plan_push_times(plan)
    s_ns, e_ns = kvx.kvx_plan_push_times_ns(plan)
    t = e - s
    assert len(t) == 4 and np.all(t > 0) and np.all(t < 1e5) and s.min() == 0
    assert np.allclose((e_ns - s_ns) * 1e-3, t, atol=0.01) and np.all(s_ns > 0)
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(4))
    # a second round: fresh slots, stamped later on the same clock
    assert push_all_layers(plan, 4) == kvx.KVX_OK
    s2_ns, e2_ns = kvx.kvx_plan_push_times_ns(plan)
    assert len(s2_ns) == 4 and s2_ns.min() > e_ns.max() and np.all(e2_ns > s2_ns)
    kvx.kvx_plan_destroy(plan)


def test_timing_plan_with_nothing_to_copy_has_no_entries():
    w = kvx_inputs.tiny()
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), [], {"flags": kvx.KVX_PLAN_TIMING})
    assert push_all_layers(plan, w.src.n_layers) == kvx.KVX_OK
    assert len(kvx.kvx_plan_push_times(plan)[0]) == 0 and len(kvx.kvx_plan_push_times_ns(plan)[0]) == 0
    kvx.kvx_plan_destroy(plan)


def test_notify_event_orders_a_consumer_stream():
    """A consumer stream that waits on the push's notification event sees the pushed layer."""
    w = kvx_inputs.qwen3_32b_single(n_layers=3)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    side, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in range(3)]
    copies = []
    for layer in range(3):
        kvx.kvx_push_layer_notify(plan, layer, layer + 1, side, None, done[layer])
        consumer.wait_event(done[layer])
        with torch.cuda.stream(consumer):
            copies.append([b.clone() for b in layer_buffers(w.dst, dst, layer)])
    consumer.synchronize()
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    for layer in range(3):
        for a, b in zip(copies[layer], layer_buffers(w.dst, dst, layer)):
            assert torch.equal(a, b)
    kvx.kvx_plan_destroy(plan)


def test_set_opts_on_existing_plan():
    w = kvx_inputs.qwen3_32b_batched(n_layers=2, n_requests=3)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w))
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    kvx.kvx_plan_set_opts(plan, {"flags": kvx.KVX_PLAN_TIMING, "kernel": kvx.KVX_KERNEL_BULK, "lanes": 1})
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_BULK
    assert push_all_layers(plan, 2) == kvx.KVX_OK
    s, e = kvx.kvx_plan_push_times(plan)
    assert len(s) == 2 and np.all(e > s)
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(2))
    kvx.kvx_plan_destroy(plan)


def test_hnd_batched_workload_sampled():
    """The batched Qwen3-32B-shaped workload with both pools head-major, 64 layers, sampled layers."""
    w = kvx_inputs.qwen3_32b_batched_hnd()
    info = run_workload(w, [0, 40, 63])
    assert info["strided"] == 1 and info["src_pitch"] == 256 and info["dst_pitch"] == 256


@pytest.mark.parametrize("kernel", ["auto", "tensor", "staged"])
@pytest.mark.parametrize("name", ["qwen3_32b_single_nhd_to_hnd", "qwen3_32b_single_hnd_to_nhd"])
def test_head_layout_change_per_layer_full_size(name, kernel):
    """The per-layer head-layout changes at full size (64 layers, one 8192-token request, 32 MiB a
    layer) in the benchmark's launch pattern: the automatic kernel (tensor-map copies), and staged."""
    w = kvx_inputs.PUSH_WORKLOADS[name]()
    info = run_workload(w, [0, 31, 63], opts={"kernel": KERNELS.get(kernel, 0)})
    assert info["kernel"] == (kvx.KVX_KERNEL_STAGED if kernel == "staged" else kvx.KVX_KERNEL_TENSOR)


@pytest.mark.parametrize("kernel", ["tensor", "staged"])
def test_head_layout_stall_reports_failed(kernel):
    """The stall hook on a head-layout-changing plan: the waiting CTA gives up, the layer reads FAILED,
    layers read DONE only when exact, and a second push completes."""
    w = kvx_inputs.qwen3_32b_single_nhd_to_hnd(n_layers=3)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w), {"kernel": KERNELS[kernel]})
    assert kvx.kvx_plan_get_info(plan)["kernel"] == KERNELS[kernel]
    side = torch.cuda.Stream()
    kvx.kvx_plan_inject_stall(plan, 2)
    for layer in range(3):
        kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_EFAILED
    states = kvx.kvx_plan_layer_states(plan).tolist()
    assert states == [kvx.KVX_LAYER_DONE, kvx.KVX_LAYER_DONE, kvx.KVX_LAYER_FAILED]
    assert_layer_states_truthful(w, src, dst, states, kvx_inputs.CANARY_BF16)
    kvx.kvx_push_layer(plan, 2, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(3))
    kvx.kvx_plan_destroy(plan)


def test_nhd_to_hnd_batched_workload_sampled():
    """The batched Qwen3-32B-shaped workload from a token-major producer into a head-major consumer,
    64 layers in the benchmark's launch pattern (head-group tiles), sampled layers checked whole."""
    w = kvx_inputs.qwen3_32b_batched_nhd_to_hnd()
    info = run_workload(w, [0, 33, 63])
    assert info["strided"] == 1 and info["src_head_pitch"] == 256 and info["dst_head_pitch"] == 16 * 256


def test_threads_push_their_own_plans_concurrently():
    """kvx calls from several host threads, each with its own plan, pools and stream (the library's
    lanes, event pool, device memory pool and status stream are shared): every consumer equals the
    oracle on its producer."""
    import threading
    n_threads, reps = 4, 8
    cases = []
    for k in range(n_threads):
        w = kvx_inputs.qwen3_32b_batched(seed=40 + k, n_layers=3, n_requests=3, len_range=(200, 1500))
        src, _ = device_pool(w.src, w.values, seed=w.seed + k)
        dst, _ = device_pool(w.dst, "canary_" + w.values)
        cases.append((w, src, dst))
    errors = []

    def worker(k):
        try:
            w, src, dst = cases[k]
            stream = torch.cuda.Stream()
            for _ in range(reps):
                plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w),
                                       {"flags": kvx.KVX_PLAN_TIMING if k % 2 else 0})
                for layer in range(w.src.n_layers):
                    kvx.kvx_push_layer(plan, layer, stream)
                assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
                kvx.kvx_plan_destroy(plan)
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for w, src, dst in cases:
        per = w.dst.n_planes * w.dst.n_shards
        check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(per)],
                     reqs_of(w), range(w.src.n_layers))


def assert_layer_states_truthful(w, src, dst, states, canary_elem):
    """A layer that reads DONE equals the oracle byte for byte; a FAILED one holds, element by element,
    either the oracle's value or its prior canary (nothing outside the pushed tokens moved)."""
    orc = oracle.load()
    sg1, dg1 = w.src.replace(n_layers=1), w.dst.replace(n_layers=1)
    for layer, st in enumerate(states):
        want = [canary_host(w.dst, w.values) for _ in range(w.dst.n_planes * w.dst.n_shards)]
        orc.push(sg1, host(layer_buffers(w.src, src, layer)), dg1, want, reqs_of(w))
        got = host(layer_buffers(w.dst, dst, layer))
        for a, b in zip(got, want):
            if st == kvx.KVX_LAYER_DONE:
                assert np.array_equal(a, b), f"layer {layer} reads DONE but differs from the oracle"
            else:
                a16, b16 = a.view(np.uint16), b.view(np.uint16)
                assert bool(((a16 == b16) | (a16 == canary_elem)).all()), f"layer {layer}: a byte moved outside the push"


@pytest.mark.parametrize("multi_layer", [False, True], ids=["per_layer", "one_launch"])
def test_bulk_wait_runs_out_and_reports_failed(multi_layer):
    """kvx_plan_inject_stall: the bulk kernel's first CTA waits, after a stage's loads landed, for a
    phase of that stage that nothing arms. The wait gives up at the hook's 1 ms limit (no hang, no
    fault), every layer of the work that CTA had left reads FAILED at kvx_sync, layers read DONE only
    when exact, and no consumer byte outside the pushed tokens changes. The hook fires once: the next
    push of the same layers is complete and exact."""
    w = kvx_inputs.qwen3_32b_single(n_layers=3)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    opts = {"layers_per_launch": 3} if multi_layer else None
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w), opts)
    assert kvx.kvx_plan_get_info(plan)["kernel"] == kvx.KVX_KERNEL_BULK
    side = torch.cuda.Stream()
    if multi_layer:
        kvx.kvx_plan_inject_stall(plan, 0)
        kvx.kvx_push_layers(plan, 0, 3, side)
    else:
        kvx.kvx_plan_inject_stall(plan, 1)
        for layer in range(3):
            kvx.kvx_push_layer(plan, layer, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_EFAILED
    states = kvx.kvx_plan_layer_states(plan).tolist()
    if multi_layer:
        # the stalled CTA held work in every layer of the one launch: all three are reported
        assert states == [kvx.KVX_LAYER_FAILED] * 3
    else:
        assert states == [kvx.KVX_LAYER_DONE, kvx.KVX_LAYER_FAILED, kvx.KVX_LAYER_DONE]
    assert_layer_states_truthful(w, src, dst, states, kvx_inputs.CANARY_BF16)
    # the hook fired once
    if multi_layer:
        kvx.kvx_push_layers(plan, 0, 3, side)
    else:
        kvx.kvx_push_layer(plan, 1, side)
    assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(2)], reqs_of(w),
                 range(3))
    kvx.kvx_plan_destroy(plan)


def test_stall_hook_needs_the_bulk_kernel():
    w = kvx_inputs.tiny()
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    plan = kvx.kvx_plan_ex(kvx.Pool(w.src, src), kvx.Pool(w.dst, dst), reqs_of(w), {"kernel": KERNELS["persist"]})
    with pytest.raises(kvx.KvxError) as ei:
        kvx.kvx_plan_inject_stall(plan, 0)
    assert ei.value.status == kvx.KVX_EUNSUPPORTED
    kvx.kvx_plan_destroy(plan)


@pytest.mark.parametrize("lookahead,all_layers", [(1, 0), (2, 0), (3, 1)])
def test_native_engine_loop_pushes_exact_bytes(lookahead, all_layers):
    """The benchmark's native engine loop (kvx_fixture_run_steps: a plan per step, per layer the prefill
    fixture and the gated push, `lookahead` steps in flight, timing plans every other step) leaves the
    consumer pool equal to the oracle's push on every layer, with every plan synced and destroyed."""
    import ctypes
    w = kvx_inputs.qwen3_32b_single(n_layers=4)
    src, _ = device_pool(w.src, w.values, seed=w.seed)
    dst, _ = device_pool(w.dst, "canary_" + w.values)
    sp, dp = kvx.Pool(w.src, src), kvx.Pool(w.dst, dst)
    carr, n_req, _keep = kvx._requests(reqs_of(w))
    o = kvx._opts({})
    main, side = torch.cuda.Stream(priority=-1), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(w.src.n_layers)]
    for ev in ready:
        ev.record(main)
    ready_arr = (ctypes.c_void_p * w.src.n_layers)(*[int(ev.cuda_event) for ev in ready])
    cap = 4096
    s_ns, e_ns = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
    n_st = ctypes.c_int64(0)
    n_steps = 5
    iss, pln = np.zeros(n_steps), np.zeros(n_steps)
    fx = prefill_fixture.lib()
    rc = fx.kvx_fixture_run_steps(ctypes.addressof(sp.struct), ctypes.addressof(dp.struct), ctypes.addressof(carr),
                                  n_req, ctypes.addressof(o), 2, n_steps, all_layers, 8, 2000, int(main.cuda_stream),
                                  int(side.cuda_stream), ctypes.addressof(ready_arr), None, s_ns.ctypes.data,
                                  e_ns.ctypes.data, cap, ctypes.addressof(n_st), iss.ctypes.data, pln.ctypes.data,
                                  lookahead)
    assert rc == 0, fx.kvx_fixture_last_error().decode()
    torch.cuda.synchronize()
    assert n_st.value > 0 and (e_ns[:n_st.value] >= s_ns[:n_st.value]).all()   # timed steps carry stamps
    per = w.dst.n_planes * w.dst.n_shards
    check_layers(w.src, src, w.dst, dst, lambda l: [canary_host(w.dst, w.values) for _ in range(per)],
                 reqs_of(w), range(w.src.n_layers))
