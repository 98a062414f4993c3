"""CPU tests of the benchmark's host logic: the multi-rank reduction (gloo, world size 2), the
reference arm (the oracle timed on the host) alone and under torchrun, and interval union."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

torch = pytest.importorskip("torch")


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, n = bench.reduce_over_ranks(elapsed_ms=10.0 + 5 * rank, launches=100 + rank, device="cpu")
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump([t, n], f)
    dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path / "r")), nprocs=2, start_method="spawn")
    for r in range(2):
        t, n = json.load(open(tmp_path / f"r.{r}"))
        assert t == 15.0 and n == 201              # max of the times, sum of the launches


def test_union_of_intervals():
    s = np.array([0.0, 5.0, 20.0, 22.0], np.float32)
    e = np.array([10.0, 12.0, 25.0, 23.0], np.float32)
    assert bench.union_us(s, e) == pytest.approx(17.0)
    assert bench.union_us(np.zeros(0, np.float32), np.zeros(0, np.float32)) == 0.0


def run_bench(args, env=None):
    r = subprocess.run([sys.executable, *args], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, **(env or {})})
    assert r.returncode == 0, r.stderr[-3000:]
    return r


def test_reference_arm_single_process():
    r = run_bench(["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"] == bench.METRIC


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    r = run_bench(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
                   "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2",
                   "--steps", "1", "--warmup", "3"])
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_clock_by_step_bins_and_nearest_sample():
    fine = [(10.0000, 2070.0), (10.0021, 1980.0), (10.0100, 1500.0)]
    steps = [9.9990, 10.0005, 10.0011, 10.0030, 10.0400, 10.0500]
    got = bench.clock_by_step(fine, steps)
    # step 0 holds the first sample; steps 1 and 2 take the nearest one (within 3 ms of their middle);
    # step 3 holds the last sample; step 4's middle is 35 ms from every sample
    assert got == [2070.0, 2070.0, 1980.0, 1500.0, None]
    assert bench.clock_by_step([], steps) == [None] * 5
