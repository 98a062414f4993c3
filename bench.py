"""Benchmark of the kvx layer push (and, on rank 0, the end-to-end path, the prefix match, the
prefill/push overlap, the other push configurations and the oracle on the host's cores).

Default workload: the Qwen3-32B-shaped single-request push (64 layers x {K,V}, 8 KV heads x 128 bf16,
block 16, one 8192-token prompt = 512 blocks, pools of 615 blocks, destination ids chunked).

One step = the whole push path for one batch of requests on the workload's pools: build the plan,
then per layer run the synthetic prefill fixture on the priority stream (it records the layer's
ready event) and kvx_push_layer gated on that event. Steps are issued with two steps of look-ahead (a
step's plan is synced after the two steps after it have been issued). The pools are far larger than L2, so no
flush is needed between steps.

value = read+write bytes of all timed steps / device time of the timed steps (CUDA events on the
prefill stream around all steps), summed over ranks / max over ranks.
roofline.achieved = the same bytes per push launch / the mean push duration, where the push
durations are the copy kernels' own global-timer stamps (first CTA start, last CTA end) and the mean
is the union of all timed launches on that one device clock / launches.
e2e = the same metric with the producer KV starting in pinned host memory and the pushed consumer
blocks gathered on the device and read back every step (per-layer copies overlapped with the pushes).

Also reported: per_config (the batched, remap, head-major and token-major -> head-major workloads,
the batched one also as a single kvx_push_layers call per step), overlap (the push beside a short
ALU prefill, a long one and a tensor-core GEMM prefill), match (block hashing, full and incremental;
the prefix-match decision with and without hole filling; the device-built pull plan and one layer
of its push), connector (requests per second through the host protocol), memcpy_ceiling and
cpu_baseline.

--impl reference times the CPU oracle instead (rank 0 only), on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(1, os.path.join(ROOT, "tests"))   # the synthetic prefill fixture lives beside the tests

import kvx_inputs  # noqa: E402
import prefill_fixture  # noqa: E402

METRIC = "KV push GB/s (read+write) and % of GB300 HBM roofline; blocks/s; prefix-match ops/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="kvx", choices=["kvx", "reference"])
    p.add_argument("--workload", default="qwen3_32b_single", choices=sorted(kvx_inputs.PUSH_WORKLOADS))
    p.add_argument("--layers", type=int, default=0,
                   help="build the workload with this many layers (0: its own count); for small profiling captures")
    p.add_argument("--tile-bytes", type=int, default=0)
    p.add_argument("--threads", type=int, default=0)
    p.add_argument("--kernel", type=int, default=0, help="KVX_KERNEL_*: 0 auto, 1 tile, 2 persist, 3 bulk, 4 tensor, 5 staged")
    p.add_argument("--max-ctas", type=int, default=0, help="upper bound on the CTAs of one copy launch (0: none)")
    p.add_argument("--ctas-per-sm", type=int, default=0)
    p.add_argument("--lanes", type=int, default=0, help="internal push streams (0: library default)")
    p.add_argument("--bulk-stages", type=int, default=0, help="bulk kernel ring stages (0: library default)")
    p.add_argument("--lookahead", type=int, default=2,
                   help="engine loop: steps issued before the oldest one is synced (1: sync a step after the next is issued)")
    p.add_argument("--fixture-ctas", type=int, default=8)
    p.add_argument("--fixture-iters", type=int, default=2000)
    p.add_argument("--timing-every", type=int, default=4,
                   help="time the pushes of every n-th timed step only (1: every step; reading the stamps "
                        "back costs the host about 25 us per timed step)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--cpu-config-seconds", type=float, default=4.0,
                   help="oracle time on each other configuration (all cores, then one)")
    p.add_argument("--no-match", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="skip the short runs of the other push configs")
    p.add_argument("--no-overlap", action="store_true", help="skip the prefill / push overlap measurement")
    p.add_argument("--overlap-narrow", default="32:6,64:4",
                   help="push shapes beside the GEMM prefill, separated by commas: max_ctas:bulk_stages pairs, "
                        "or plan options as key=value;key=value")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes of the push kernel from a committed ncu summary, if the kernel source is
    unchanged since the capture (else None)."""
    rec = None
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("csrc_sha") != csrc_sha():
        return None
    return rec.get("dram_bytes_per_launch")


def csrc_sha():
    """Hash of the code of the copy kernels and the copy-shape builder, comments and blank space left
    out (the ncu counters are valid only for this code)."""
    h = hashlib.sha256()
    for name in ("kvx_copy.cu", "kvx_tiles.cpp"):
        with open(os.path.join(ROOT, "disaggregated_prefill_decode_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def requests(w):
    return [(r.n_tokens, r.src_ids, r.dst_ids) for r in w.requests]


def union_us(start, end):
    """Length of the union of intervals [start_i, end_i]."""
    total, cur_s, cur_e = 0.0, None, None
    for s, e in sorted(zip(start.tolist(), end.tolist())):
        if cur_e is None or s > cur_e:
            if cur_e is not None:
                total += cur_e - cur_s
            cur_s, cur_e = s, e
        else:
            cur_e = max(cur_e, e)
    if cur_e is not None:
        total += cur_e - cur_s
    return total


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------

# The SM clock read through NVML every 2 ms in a child process (its own interpreter, so the sampling
# takes nothing from the issuing thread), each sample stamped with the host's monotonic clock: fine
# enough to tell the clock of each step of a short timed region.
_NVML_POLLER = r"""
import ctypes, sys, time
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(1)
h = ctypes.c_void_p()
if nv.nvmlDeviceGetHandleByUUID(sys.argv[1].encode(), ctypes.byref(h)) != 0:
    sys.exit(1)
clk = ctypes.c_uint()
out = sys.stdout
while True:
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:        # 1: the SM clock
        out.write(f"{time.monotonic():.6f} {clk.value}\n")
    time.sleep(0.002)
"""


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid):
        self.proc = None
        self.fine = None
        self.uuid = device_uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.uuid:
            try:
                self.fine = subprocess.Popen([sys.executable, "-u", "-c", _NVML_POLLER, self.uuid], stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.fine = None

    def stop_fine(self):
        """(host monotonic time, SM MHz) samples of the NVML poller, or []."""
        if not self.fine:
            return []
        self.fine.terminate()
        out, _ = self.fine.communicate(timeout=10)
        samples = []
        for line in out.splitlines():
            parts = line.split()
            if len(parts) == 2:
                try:
                    samples.append((float(parts[0]), float(parts[1])))
                except ValueError:
                    pass
        return samples

    def stop(self):
        fine = self.stop_fine()
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0,
                    "fine": fine}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "fine": fine}


def clock_by_step(fine, step_host, reach_s=0.003):
    """NVML SM clock per timed step: the median of the samples inside the step's host issue window
    [start_i, start_{i+1}), else the sample nearest the window's middle if one lies within reach_s
    (samples come every few ms, steps last under one), else None. The GPU runs up to a step behind
    the host, so this places clocks to within a step or two."""
    out = []
    for a, b in zip(step_host[:-1], step_host[1:]):
        v = [mhz for t, mhz in fine if a <= t < b]
        if v:
            out.append(statistics.median(v))
            continue
        mid = 0.5 * (a + b)
        near = min(fine, key=lambda x: abs(x[0] - mid), default=None)
        out.append(near[1] if near is not None and abs(near[0] - mid) <= reach_s else None)
    return out


# ---------------------------------------------------------------------------------------------
# kvx arm
# ---------------------------------------------------------------------------------------------

def alloc_pool(torch, geom, fill, seed, device):
    per = -(-geom.buffer_bytes // 512) * 512
    big = torch.empty(per * geom.n_buffers, dtype=torch.uint8, device=device)
    if fill == "src":
        kvx_inputs.fill_bf16_normal(big, seed) if geom.elem_bytes == 2 else kvx_inputs.fill_fp8_bytes(big, seed)
    else:
        kvx_inputs.fill_canary(big, "bf16_normal" if geom.elem_bytes == 2 else "fp8_bytes")
    torch.cuda.synchronize(device)   # filled on the current stream; the pushes run on others
    return [big[i * per:i * per + geom.buffer_bytes] for i in range(geom.n_buffers)], big


def time_push_workload(args, torch, kvx, w, device, K, W, every, sampler=None, barrier=None, all_layers=False,
                       extra_opts=None):
    """Allocates the workload's pools and times K steps of the per-layer push pattern after W untimed
    ones. A step builds the requests' plan, runs the synthetic prefill (per layer a fixture kernel on
    the priority stream that records the layer's ready event) and pushes every layer gated on its
    event; each step is synced after `args.lookahead` later steps are issued. The pushes of every `every`-th step are
    timed (the kernels' own global-timer stamps); the warm-up steps follow the same pattern, so the
    timed loop meets no first use. `all_layers`: one kvx_push_layers call per step for all layers,
    gated on the last layer's event, instead of one kvx_push_layer per layer; `extra_opts` are added
    to the plan options. `sampler` (clock sampling, started by the caller before the pools are
    allocated, since it takes a moment to start) is stopped after the timed steps; nothing idles the
    GPU between the warm-up and the timed steps."""
    L = w.src.n_layers
    src, _ = alloc_pool(torch, w.src, "src", w.seed, device)
    dst, _ = alloc_pool(torch, w.dst, "dst", 0, device)
    sp, dp = kvx.Pool(w.src, src), kvx.Pool(w.dst, dst)
    reqs = requests(w)
    opts = {"tile_bytes": args.tile_bytes, "threads": args.threads, "kernel": args.kernel,
            "ctas_per_sm": args.ctas_per_sm, "lanes": args.lanes, "bulk_stages": args.bulk_stages,
            "max_ctas": args.max_ctas}
    opts.update(extra_opts or {})
    # the synthetic prefill is the latency-critical path: its stream outranks the push stream, so the
    # copies fill the SMs the compute leaves free
    main = torch.cuda.Stream(priority=-1)
    side = torch.cuda.Stream(priority=0)
    torch.cuda.set_stream(main)

    probe = kvx.kvx_plan_ex(sp, dp, reqs, opts)
    info = kvx.kvx_plan_get_info(probe)
    kvx.kvx_plan_destroy(probe)
    ready = [torch.cuda.Event() for _ in range(L)]
    for ev in ready:                                  # materialise the events so their handles exist
        ev.record(main)
    ready_h = [int(ev.cuda_event) for ev in ready]
    main_h, side_h = int(main.cuda_stream), int(side.cuda_stream)
    fx = prefill_fixture.lib()                        # the synthetic prefill and the native engine loop
    carr, n_req, _keep = kvx._requests(reqs)
    o = kvx._opts(opts)
    cap = 4096 * 64
    s_ns, e_ns = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
    n_st = ctypes.c_int64(0)
    ready_arr = (ctypes.c_void_p * L)(*ready_h)

    def run_steps(n, timed):
        """n steps of the engine loop, natively (the fixture library's kvx_fixture_run_steps, through the
        kvx C-ABI): per step a plan (a timing plan when the step's index is a multiple of `every`, the
        warm-up steps included, so the timed loop meets no first use), per layer the fixture and the
        gated push; each step synced after `args.lookahead` later ones are issued. Timed runs record a CUDA event on
        the prefill stream where each step starts and after the last sync."""
        marks, marks_arr = None, None
        if timed:
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            for m in marks:                           # materialise the handles
                m.record(main)
            torch.cuda.synchronize()
            marks_arr = (ctypes.c_void_p * (n + 1))(*[int(m.cuda_event) for m in marks])
        iss, pln = np.zeros(max(n, 1)), np.zeros(max(n, 1))
        rc = fx.kvx_fixture_run_steps(ctypes.addressof(sp.struct), ctypes.addressof(dp.struct), ctypes.addressof(carr),
                                      n_req, ctypes.addressof(o), every, n, int(all_layers), args.fixture_ctas,
                                      args.fixture_iters, main_h, side_h, ctypes.addressof(ready_arr),
                                      ctypes.addressof(marks_arr) if timed else None,
                                      s_ns.ctypes.data if timed else None, e_ns.ctypes.data if timed else None, cap,
                                      ctypes.addressof(n_st), iss.ctypes.data, pln.ctypes.data, args.lookahead)
        if rc:
            raise RuntimeError(f"engine loop: {fx.kvx_fixture_last_error().decode()}")
        return marks, iss[:n], pln[:n]

    gc.collect()
    gc.disable()                                      # no collector pauses in the warm-up or the timed loop
    run_steps(W, False)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    launches0 = kvx.kvx_launch_count() + prefill_fixture.launch_count()
    torch.cuda.synchronize()
    host0 = time.monotonic()
    wall0 = time.perf_counter()
    step_marks, issue_us, plan_us = run_steps(K, True)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = sampler.stop() if sampler else None
    gc.enable()
    launches = kvx.kvx_launch_count() + prefill_fixture.launch_count() - launches0
    step_host = np.concatenate([[0.0], np.cumsum(issue_us)]) * 1e-6 + host0
    push_times = [(s_ns[:n_st.value], e_ns[:n_st.value])]
    t0, t1 = step_marks[0], step_marks[-1]
    step_ms = [a.elapsed_time(b) for a, b in zip(step_marks[:-1], step_marks[1:])]
    # Pushes of consecutive layers (and of consecutive steps) may overlap: they run on separate lanes.
    # The kernels stamp the GPU's one global timer, so all timed pushes share a timeline; the time the
    # GPU spends pushing is the union of their intervals, per launch that union / launches.
    all_s = np.concatenate([s_ns for s_ns, _ in push_times])
    all_e = np.concatenate([e_ns for _, e_ns in push_times])
    t_base = all_s.min()                              # int64 first: the timer's epoch is far from zero
    all_s, all_e = (all_s - t_base) * 1e-3, (all_e - t_base) * 1e-3
    busy_us = union_us(all_s, all_e)
    raw_us = (all_e - all_s).tolist()
    timed_step_ms = sum(step_ms[i] for i in range(0, K, every))
    torch.cuda.set_stream(torch.cuda.default_stream(device))
    return {"w": w, "L": L, "src": src, "dst": dst, "sp": sp, "dp": dp, "reqs": reqs, "opts": opts, "info": info,
            "bytes_step": 2 * info["bytes_per_layer"] * L,                     # read + write
            "blocks_step": sum(-(-n // w.src.block_size) for n, _, _ in reqs) * L,
            "elapsed_ms": t0.elapsed_time(t1), "launches": launches, "clocks": clk, "wall": wall,
            "timed_steps": -(-K // every), "timed_launches": len(raw_us),
            "mean_push_ms": busy_us / len(raw_us) * 1e-3,
            "raw_push_ms": statistics.fmean(raw_us) * 1e-3,
            "step_ms": step_ms, "push_cover": busy_us * 1e-3 / timed_step_ms,
            "step_host": step_host.tolist(),
            "issue_us": issue_us.tolist(), "plan_us": plan_us.tolist()}


def measure_overlap(args, torch, kvx, m, steps=200):
    """The pages' premise, measured: is the push off the prefill's critical path? Per step, the
    synthetic prefill alone (the L fixture launches on the priority stream), the pushes alone (the L
    layer pushes, no gate), and both (the benchmark's pattern: each push gated on its layer's event);
    and how long the prefill chain itself takes inside the combined run. Three times: with the
    benchmark's fixture (a prefill layer shorter than its push), with one 8 times longer (a prefill
    layer longer than its push, the regime of a real model, whose layers take far longer than their KV
    copy), and with layers of tensor-core work (one bf16 GEMM each) instead of the ALU fixture."""
    L, reqs, sp, dp = m["L"], m["reqs"], m["sp"], m["dp"]
    opts = m["opts"]
    lib = kvx._lib
    fx = prefill_fixture.lib().kvx_fixture_prefill
    main = torch.cuda.Stream(priority=-1)
    side = torch.cuda.Stream(priority=0)
    ready = [torch.cuda.Event() for _ in range(L)]
    for ev in ready:
        ev.record(main)
    ready_h = [int(ev.cuda_event) for ev in ready]
    main_h, side_h = int(main.cuda_stream), int(side.cuda_stream)

    # a prefill layer made of tensor-core work instead of the ALU fixture: one bf16 GEMM of the
    # layer's 8192 tokens by a 5120 x 5120 weight (a Qwen3-32B attention projection)
    gemm = [torch.randn(8192, 5120, dtype=torch.bfloat16, device=main.device),
            torch.randn(5120, 5120, dtype=torch.bfloat16, device=main.device)]
    gemm.append(torch.empty(8192, 5120, dtype=torch.bfloat16, device=main.device))
    torch.cuda.synchronize()

    def run(prefill, push, n, iters, push_opts=None):
        prev, marks = None, []
        for _ in range(n):
            plan = kvx.kvx_plan_ex(sp, dp, reqs, dict(opts, **(push_opts or {}))) if push else None
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for layer in range(L):
                if prefill and iters < 0:
                    with torch.cuda.stream(main):
                        torch.matmul(gemm[0], gemm[1], out=gemm[2])
                        ready[layer].record(main)
                elif prefill:
                    fx(args.fixture_ctas, iters, None, 0, layer, main_h, ready_h[layer])
                if push:
                    lib.kvx_push_layer(plan.handle, layer, side_h, ready_h[layer] if prefill else None)
            b.record(main)
            marks.append((a, b))
            if prev is not None:
                assert kvx.kvx_sync(prev, -1) == kvx.KVX_OK
                kvx.kvx_plan_destroy(prev)
            prev = plan
        if prev is not None:
            assert kvx.kvx_sync(prev, -1) == kvx.KVX_OK
            kvx.kvx_plan_destroy(prev)
        return marks

    def timed(prefill, push, iters, n_steps=steps, push_opts=None):
        run(prefill, push, 3, iters, push_opts)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        marks = run(prefill, push, n_steps, iters, push_opts)
        main.wait_stream(side)
        t1.record(main)
        torch.cuda.synchronize()
        chain = statistics.median(a.elapsed_time(b) for a, b in marks) if prefill else None
        return t0.elapsed_time(t1) / n_steps, chain

    def interleaved(push_opts, iters=-1, n_pairs=24):
        """Prefill steps (GEMM layers for iters < 0, else the ALU fixture) alternating without and with
        the pushes, each step on its own (the GPU drained before the next), so clock and power drift
        falls on both alike: the median chain time of each kind, and of the steps with pushes the median
        span from the first layer to the end of the last copy (each lane's last push, in round-robin lane
        order the last `lanes` layers, records an event after its copy)."""
        alone, with_push, span = [], [], []
        tail = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
        for ev in tail:
            ev.record(main)                           # torch creates an event at its first record
        for i in range(2 * (n_pairs + 2)):
            push = i % 2 == 1
            plan = kvx.kvx_plan_ex(sp, dp, reqs, dict(opts, **(push_opts or {}))) if push else None
            n_tail = min(L, kvx.kvx_plan_get_info(plan)["lanes"]) if push else 0
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for layer in range(L):
                if iters < 0:
                    with torch.cuda.stream(main):
                        torch.matmul(gemm[0], gemm[1], out=gemm[2])
                        ready[layer].record(main)
                else:
                    fx(args.fixture_ctas, iters, None, 0, layer, main_h, ready_h[layer])
                if push and layer >= L - n_tail:
                    kvx.kvx_push_layer_notify(plan, layer, layer + 1, side, ready[layer], tail[layer])
                elif push:
                    lib.kvx_push_layer(plan.handle, layer, side_h, ready_h[layer])
            b.record(main)
            if push:
                assert kvx.kvx_sync(plan, -1) == kvx.KVX_OK
                kvx.kvx_plan_destroy(plan)
            torch.cuda.synchronize()
            if i >= 4:                                # the first two pairs warm up
                (with_push if push else alone).append(a.elapsed_time(b))
                if push:
                    span.append(max([a.elapsed_time(b)] + [a.elapsed_time(tail[l]) for l in range(L - n_tail, L)]))
        return statistics.median(alone), statistics.median(with_push), statistics.median(span)

    push_only, _ = timed(False, True, 0)
    out = {"push_only_ms_per_step": round(push_only, 4)}
    for name, iters in (("short_prefill", args.fixture_iters), ("long_prefill", 8 * args.fixture_iters),
                        ("gemm_prefill", -1)):
        pre_only, chain_alone = timed(True, False, iters, 50 if iters < 0 else steps)
        both, chain_with = timed(True, True, iters, 50 if iters < 0 else steps)
        out[name] = {"fixture_iters": iters if iters >= 0 else "bf16 GEMM 8192 x 5120 x 5120 per layer",
                     "prefill_only_ms_per_step": round(pre_only, 4),
                     "together_ms_per_step": round(both, 4),
                     "hidden_frac": round((pre_only + push_only - both) / min(pre_only, push_only), 3),
                     "prefill_chain_ms_alone": round(chain_alone, 4),
                     "prefill_chain_ms_with_push": round(chain_with, 4),
                     "prefill_slowdown": round(chain_with / chain_alone - 1, 4)}
        # the prefill chain's slowdown from steps alternating without and with the pushes: separate runs
        # of a chain alone drift by up to a few per cent between themselves (clock and power under a
        # 1.4 kW cap), as much as some of the effects measured, so the reported slowdown is this one
        c0, c1, sp1 = interleaved(None, iters)
        out[name]["separate_runs"] = {k: out[name][k] for k in (
            "prefill_only_ms_per_step", "together_ms_per_step", "hidden_frac", "prefill_chain_ms_alone",
            "prefill_chain_ms_with_push", "prefill_slowdown")}
        out[name].update({"prefill_chain_ms_alone": round(c0, 4), "prefill_chain_ms_with_push": round(c1, 4),
                          "prefill_slowdown": round(c1 / c0 - 1, 4), "step_ms_with_push": round(sp1, 4),
                          "hidden_frac": round((c0 + push_only - sp1) / min(c0, push_only), 3)})
        del out[name]["prefill_only_ms_per_step"], out[name]["together_ms_per_step"]
        if iters < 0:
            # the same GEMM prefill beside pushes bounded to a few CTAs with deep rings: the GEMM's CTAs
            # take every register of an SM, so each SM a copy holds is an SM the GEMM waits for
            out[name]["narrow_pushes"] = []
            variants = []
            for spec in args.overlap_narrow.split(","):
                spec = spec.strip()
                if not spec:
                    continue
                if "=" in spec:                       # key=value;key=value: any plan options
                    variants.append({k: int(v) for k, v in (kv.split("=") for kv in spec.split(";"))})
                else:                                 # max_ctas:bulk_stages
                    c, st = (int(x) for x in spec.split(":"))
                    variants.append({"max_ctas": c, "bulk_stages": st})
            for v in variants:
                p_only, _ = timed(False, True, 0, steps, v)
                c0, c1, sp1 = interleaved(v)
                out[name]["narrow_pushes"].append(
                    {"opts": v, "push_only_ms_per_step": round(p_only, 4),
                     "prefill_chain_ms_alone": round(c0, 4), "prefill_chain_ms_with_push": round(c1, 4),
                     "prefill_slowdown": round(c1 / c0 - 1, 4), "step_ms_with_push": round(sp1, 4),
                     "hidden_frac": round((c0 + p_only - sp1) / min(c0, p_only), 3)})
    out["how"] = ("24 prefill steps without and 24 with the pushes, alternating, each step drained before the "
                  "next, medians compared: the prefill chain is the time on its stream from a step's first layer to "
                  "its last, step_ms_with_push runs to the end of the last copy, prefill_slowdown = chain with / "
                  "chain alone - 1, hidden_frac = (chain alone + push alone - step with pushes) / min(chain alone, "
                  f"push alone), push alone the median of {steps} pipelined push-only steps; separate_runs: the same "
                  f"from separately timed pipelined runs ({steps} steps each, 50 with the GEMM prefill), which "
                  "drift by a few per cent between themselves (clock and power)")
    return out


def connector_rate(kvx, n=20000):
    """Requests per second through the host connector's whole protocol: registration, last prefill
    chunk, poll (READY), start, one queued write, seal, its report (all layers DONE), poll (DONE),
    release; alternate requests arrive in the other order (prefill first, deferred)."""
    import numpy as np_
    conn = kvx.kvx_conn_create()
    ids = np_.arange(16, dtype=np_.int32)
    states = np_.full(64, kvx.KVX_LAYER_DONE, np_.int32)
    t0 = time.perf_counter()
    for r in range(n):
        if r & 1:
            kvx.kvx_conn_prefill(conn, r, 0, ids, 256, True, r)
            kvx.kvx_conn_register(conn, r, 0, ids, r)
        else:
            kvx.kvx_conn_register(conn, r, 0, ids, r)
            kvx.kvx_conn_prefill(conn, r, 0, ids, 256, True, r)
        kvx.kvx_conn_poll(conn, r, 8)
        kvx.kvx_conn_start(conn, r, 0, r)
        kvx.kvx_conn_write_issued(conn, r, 0, 0, 1)
        kvx.kvx_conn_seal(conn, r, 0, 0)
        kvx.kvx_conn_write_done(conn, r, 0, 0, states, now_us=r)
        kvx.kvx_conn_poll(conn, r, 8)
        kvx.kvx_conn_release(conn, r)
    dt = time.perf_counter() - t0
    kvx.kvx_conn_destroy(conn)
    return {"requests_per_s": round(n / dt, 1), "calls_per_request": 10,
            "native_requests_per_s": connector_rate_native(),
            "how": f"{n} requests through the Python binding, one host thread: the figure is mostly the "
                   "binding's per-call cost (about 4 us a call); native_requests_per_s is the same protocol "
                   "driven from C (tests/c/kvx_conn_rate.c, built with gcc here), 200000 requests"}


def connector_rate_native():
    """The connector's protocol driven from plain C against libkvx.so; None when no C compiler."""
    import shutil
    import tempfile
    if not shutil.which("gcc"):
        return None
    pkg = os.path.join(ROOT, "disaggregated_prefill_decode_gb300")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "kvx_conn_rate")
        r = subprocess.run(["gcc", "-std=c11", "-O2", os.path.join(ROOT, "tests", "c", "kvx_conn_rate.c"), "-o", exe,
                            "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), "-L", pkg, "-lkvx",
                            "-L", os.path.join(cuda, "lib64"), "-lcudart",
                            f"-Wl,-rpath,{pkg}:{os.path.join(cuda, 'lib64')}"], capture_output=True, text=True)
        if r.returncode != 0:
            return None
        r = subprocess.run([exe, "200000"], capture_output=True, text=True, timeout=120)
        if r.returncode != 0:
            return None
        return round(float(r.stdout.split()[-1]), 1)


KERNEL_NAMES = ["kvx_copy_tiles", "kvx_copy_tiles", "kvx_copy_persist", "kvx_copy_bulk", "kvx_copy_bulk (tensor maps)",
                "kvx_copy_staged"]
KERNEL_SHORT = ["auto", "tile", "persist", "bulk", "tensor", "staged"]


def per_config(args, torch, kvx, device):
    """The other push configurations, briefly, in the same run: GB/s and blocks/s per step, the push
    kernel's roofline fraction (union of all push intervals on the kernels' global-timer stamps)."""
    peak, _ = measured_peak()
    out = []
    per_layer_call = "one kvx_push_layer call per layer, gated on its layer"
    one_call = "one kvx_push_layers call per step for all layers, after the prefill's last layer"
    cases = (("tiny", 200, False, None, per_layer_call),
             ("qwen3_32b_batched", 20, False, None, per_layer_call),
             ("qwen3_32b_batched", 20, True, None, one_call + " (default: launches of about 256 MiB on the lanes)"),
             ("qwen3_32b_batched", 20, True, {"layers_per_launch": 64}, one_call + " in a single launch"),
             ("tp4_to_tp1_remap", 20, False, None, per_layer_call),
             ("qwen3_32b_batched_hnd", 20, False, None, per_layer_call),
             ("qwen3_32b_batched_nhd_to_hnd", 20, False, None, per_layer_call),
             ("qwen3_32b_single_nhd_to_hnd", 100, False, None, per_layer_call),
             ("qwen3_32b_single_hnd_to_nhd", 100, False, None, per_layer_call))
    for name, steps, all_layers, extra, launch in cases:
        if name == args.workload and not all_layers:
            continue
        m = time_push_workload(args, torch, kvx, kvx_inputs.PUSH_WORKLOADS[name](), device, steps, 3, 1,
                               all_layers=all_layers, extra_opts=extra)
        bytes_launch = 2 * m["info"]["bytes_per_layer"] * m["L"] * m["timed_steps"] // m["timed_launches"]
        achieved = bytes_launch / (m["mean_push_ms"] * 1e-3) / 1e9
        out.append({"workload": name, "steps": steps, "launch": launch,
                    "launches_per_step": m["timed_launches"] // m["timed_steps"],
                    "value": round(m["bytes_step"] * steps / (m["elapsed_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "blocks_per_s": round(m["blocks_step"] * steps / (m["elapsed_ms"] * 1e-3), 1),
                    "roofline_frac": round(achieved / peak, 4), "mean_launch_us": round(m["mean_push_ms"] * 1e3, 3),
                    "kernel": KERNEL_NAMES[m["info"]["kernel"]], "threads": m["info"]["threads"],
                    "bytes_per_launch": bytes_launch,
                    "l2": (f"inputs larger than L2 ({m['bytes_step'] / 1e9:.2f} GB read+written per step); no flush"
                           if m["bytes_step"] > (129 << 20) else
                           f"fits in L2 ({m['bytes_step'] / 1e6:.1f} MB per step), not flushed: launch-bound, reported"),
                    "traffic": None if all_layers else ncu_traffic(name)})
        del m
        gc.collect()
        torch.cuda.empty_cache()
    out.append(bidir_full(torch, kvx, device, {"kernel": args.kernel, "threads": args.threads,
                                                "ctas_per_sm": args.ctas_per_sm, "bulk_stages": args.bulk_stages}))
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_kvx(args, rank, local_rank, world):
    import torch
    import torch.distributed as dist
    from disaggregated_prefill_decode_gb300 import kvx

    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    make = kvx_inputs.PUSH_WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    every = max(1, args.timing_every)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    m = time_push_workload(args, torch, kvx, make(n_layers=args.layers) if args.layers > 0 else make(), device,
                           K, W, every, sampler=sampler, barrier=dist.barrier if world > 1 else None)
    w, L, info, reqs = m["w"], m["L"], m["info"], m["reqs"]
    src, dst, sp, dp, opts, bytes_step = m["src"], m["dst"], m["sp"], m["dp"], m["opts"], m["bytes_step"]
    elapsed_ms, launches = m["elapsed_ms"], m["launches"]
    mean_push_ms, raw_push_ms = m["mean_push_ms"], m["raw_push_ms"]
    if world > 1:
        elapsed_ms, launches = reduce_over_ranks(elapsed_ms, launches, device)

    peak, peak_kind = measured_peak()
    achieved = 2 * info["bytes_per_layer"] / (mean_push_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(world * bytes_step * K / (elapsed_ms * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8",
        "data": "synthetic: seeded bf16 N(0,1) producer KV, consumer canary 0xDEAD, seeded chunked block ids",
        "config": {
            "workload": args.workload,
            "layers": L, "planes": w.src.n_planes,
            "producer": f"{w.src.n_shards} x [{w.src.n_blocks}][{w.src.block_size}][{w.src.heads_per_shard}][{w.src.head_dim}] x {w.src.elem_bytes} B",
            "consumer": f"{w.dst.n_shards} x [{w.dst.n_blocks}][{w.dst.block_size}][{w.dst.heads_per_shard}][{w.dst.head_dim}] x {w.dst.elem_bytes} B",
            "requests": len(reqs), "tokens": int(sum(n for n, _, _ in reqs)),
            "runs": info["n_runs"], "tiles_per_layer_plane": info["n_tiles"], "tile_bytes": info["tile_bytes"],
            "vec_bytes": info["vec_bytes"], "kernel": KERNEL_SHORT[info["kernel"]],
            "lanes": info["lanes"], "bulk_stages": info["bulk_stages"],
            "cuda_device_max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS"),
            "threads": info["threads"],
            "ctas_per_sm": args.ctas_per_sm or "auto (below 128 MiB per launch: 2 per SM on the bulk and tensor-map "
                                               "kernels, 2 persistent, 4 persistent on head groups; above: the "
                                               "occupancy limit)",
            "l2": f"inputs larger than L2: {bytes_step / 1e9:.2f} GB read+written per step vs 129 MB L2; no flush",
            "launch": f"per layer: fixture ({args.fixture_ctas} CTAs x {args.fixture_iters} iters) on a priority -1 "
                      "stream records the layer's event, then kvx_push_layer(priority 0 side stream, event) forks "
                      "onto the push lanes and waits for it; a plan is built every step and synced after "
                      f"{args.lookahead} more steps are issued; the engine loop issuing this runs natively (libkvx_fixture's "
                      "kvx_fixture_run_steps, through the kvx C-ABI)",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "blocks_per_s": round(world * m["blocks_step"] * K / (elapsed_ms * 1e-3), 1),
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
            "kernel": KERNEL_NAMES[info["kernel"]] + " (one launch per layer)",
            "raw_launch_us_mean": round(raw_push_ms * 1e3, 3),
            "timing": ("KVX_PLAN_TIMING: each copy kernel stamps the GPU global timer (first CTA start, last "
                       "CTA end) for every launch of "
                       + ("every timed step" if every == 1 else f"every {every}th timed step")
                       + "; mean_launch_us = union of all those launch intervals on that one timeline "
                       "(consecutive layers and steps overlap on the push lanes) / launches"),
            "bytes_per_launch": 2 * info["bytes_per_layer"], "mean_launch_us": round(mean_push_ms * 1e3, 3),
            "traffic": ncu_traffic(args.workload),
        },
        "gpu_launches": launches,
        "clocks": {k: v for k, v in (m["clocks"] or {}).items() if k != "fine"} or None,
        "steps_detail": step_detail(m, K),
        "host_wall_s": round(m["wall"], 4),
        "host_issue_us_per_layer": round(statistics.fmean(m["issue_us"]) / L, 3),
        "plan_build_us": round(statistics.median(m["plan_us"]), 2),
    }
    if rank == 0:
        result["memcpy_ceiling"] = memcpy_ceiling(torch, device)
        result["memcpy_ceiling"]["push_frac"] = round(achieved / result["memcpy_ceiling"]["value"], 4)
        if not args.no_overlap:
            result["overlap"] = measure_overlap(args, torch, kvx, m)
        result["connector"] = connector_rate(kvx)
        if not args.no_e2e:
            result["e2e"] = run_e2e(args, torch, kvx, w, src, dst, sp, dp, reqs, opts, bytes_step, world)
            gc.collect()
            torch.cuda.empty_cache()
            result["e2e"]["host_pools"] = run_e2e_host_pools(args, torch, kvx, w, dst, dp, reqs, opts, bytes_step)
        if not args.no_match:
            result["match"] = run_match(torch, kvx, device, {"kernel": args.kernel, "threads": args.threads,
                                                             "ctas_per_sm": args.ctas_per_sm,
                                                             "bulk_stages": args.bulk_stages})
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
            result["cpu_baseline"]["per_config"] = cpu_baseline_per_config(args.cpu_config_seconds)
        if not args.no_per_config:
            del m, src, dst, sp, dp
            result["per_config"] = per_config(args, torch, kvx, device)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def step_detail(m, K):
    """Per-step device times (CUDA events on the prefill stream where each timed step starts), the share
    of the timed steps' time in which a push kernel was running, and the SM clock per step."""
    ms = m["step_ms"]
    fine = (m["clocks"] or {}).get("fine") or []
    by_step = clock_by_step(fine, m["step_host"]) if fine else []
    return {"median_ms": round(statistics.median(ms), 5), "first_ms": round(ms[0], 5),
            "min_ms": round(min(ms), 5), "max_ms": round(max(ms), 5),
            "ms": [round(x, 4) for x in ms] if K <= 64 else None,
            "push_cover": round(m["push_cover"], 4),
            "sm_mhz_by_step": by_step if K <= 64 else None,
            "sm_mhz_fine_median": statistics.median(v for _, v in fine) if fine else None,
            "sm_mhz_fine_min": min(v for _, v in fine) if fine else None,
            "fine_samples": len(fine),
            "how": "step i = CUDA event at the start of step i+1 (or the end event) - event at the start of step i, "
                   "on the prefill stream; push_cover = union of the timed steps' push intervals / their step "
                   "time; SM clock from NVML every 2 ms, binned by each step's host issue window"}


def reduce_over_ranks(elapsed_ms, launches, device):
    """Replicas: the job's time is the slowest rank's, its launches the sum over ranks."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([launches], dtype=torch.int64, device=device)
    dist.all_reduce(n)
    dist.barrier()
    return float(t.item()), int(n.item())


def memcpy_ceiling(torch, device):
    """cudaMemcpyAsync-class device-to-device copy of 2 GiB (torch copy_), read+write GB/s; and, as the
    same kind of yardstick for head-layout changes, torch's own copy of 2 GiB of whole Qwen3-32B-shaped
    blocks from token-major to head-major ([block][16][8][128] -> [block][8][16][128], bf16)."""
    n = 1 << 31
    a = torch.empty(n, dtype=torch.uint8, device=device)
    b = torch.empty(n, dtype=torch.uint8, device=device)
    a.fill_(1)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def best_of(fn, reps=10):
        for _ in range(3):
            fn()
        best = float("inf")
        for _ in range(reps):
            s.record()
            fn()
            e.record()
            e.synchronize()
            best = min(best, s.elapsed_time(e))
        return best

    plain = best_of(lambda: b.copy_(a))
    blocks = n // (16 * 8 * 128 * 2)
    src = a.view(torch.bfloat16).view(blocks, 16, 8, 128)
    dst = b.view(torch.bfloat16).view(blocks, 8, 16, 128)
    xpose = best_of(lambda: dst.copy_(src.permute(0, 2, 1, 3)))
    del a, b, src, dst
    return {"value": round(2 * n / (plain * 1e-3) / 1e9, 1), "unit": "GB/s", "how": "torch copy_ of 2 GiB, best of 10",
            "head_transpose": {"value": round(2 * n / (xpose * 1e-3) / 1e9, 1), "unit": "GB/s",
                               "how": "torch copy_ of 2 GiB of [block][16][8][128] bf16 into [block][8][16][128] "
                                      "(token-major -> head-major whole blocks), best of 10"}}


def run_e2e_host_pools(args, torch, kvx, w, dst, dp, reqs, opts, bytes_step):
    """The end-to-end path through the C-ABI with host buffers and no separate copies: the producer
    pool lives in pinned host memory and kvx_push_layer reads it over the chip-to-chip link into the
    device consumer pool; a second plan gathers the pushed consumer blocks into a staging pool in pinned
    host memory (the kernels write it over the link). Per layer push then gather, gated by an event;
    plans built each step and synced after the next step is issued; host wall clock. The staged bytes
    must equal the producer's for the first request (equal layouts), which is checked."""
    L = w.src.n_layers
    nb = [-(-n // w.dst.block_size) for n, _, _ in reqs]
    off = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
    stage_geom = w.dst.replace(n_blocks=int(off[-1]))
    stage_reqs = [(n, d[:k], np.arange(off[i], off[i] + k, dtype=np.int32))
                  for i, ((n, _, d), k) in enumerate(zip(reqs, nb))]
    ps = -(-w.src.buffer_bytes // 4096) * 4096
    pd = -(-stage_geom.buffer_bytes // 4096) * 4096
    hsrc_big = torch.empty(ps * w.src.n_buffers, dtype=torch.uint8, pin_memory=True)
    hdst_big = torch.empty(pd * stage_geom.n_buffers, dtype=torch.uint8, pin_memory=True)
    hsrc = [hsrc_big[i * ps:i * ps + w.src.buffer_bytes] for i in range(w.src.n_buffers)]
    hdst = [hdst_big[i * pd:i * pd + stage_geom.buffer_bytes] for i in range(stage_geom.n_buffers)]
    g = torch.Generator(device=dst[0].device).manual_seed(w.seed)
    for h in hsrc:                                    # seeded bytes, drawn on the device, copied over
        h.copy_(torch.randint(0, 256, (h.numel(),), dtype=torch.uint8, device=dst[0].device, generator=g))
    hp, hs = kvx.Pool(w.src, hsrc), kvx.Pool(stage_geom, hdst)
    side = torch.cuda.Stream(priority=-1)
    ev_p = [torch.cuda.Event() for _ in range(L)]
    for ev in ev_p:
        ev.record(side)

    def issue():
        plan = kvx.kvx_plan_ex(hp, dp, reqs, opts)
        gather = kvx.kvx_plan_ex(dp, hs, stage_reqs, opts)
        for layer in range(L):
            kvx.kvx_push_layer_notify(plan, layer, layer + 1, side, None, ev_p[layer])
            kvx.kvx_push_layer(gather, layer, side, ev_p[layer])
        return plan, gather

    def finish(plans):
        for pl in plans:
            assert kvx.kvx_sync(pl, -1) == kvx.KVX_OK
            kvx.kvx_plan_destroy(pl)

    def run(n):
        prev = None
        for _ in range(n):
            cur = issue()
            if prev is not None:
                finish(prev)
            prev = cur
        finish(prev)

    run(2)
    torch.cuda.synchronize()
    t = time.perf_counter()
    run(args.e2e_steps)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t) / args.e2e_steps
    n0, b0 = int(reqs[0][0]), [int(x) for x in reqs[0][1]]
    checked = None
    if w.src.layout == w.dst.layout == kvx_inputs.LAYOUT_NHD and w.src.block_size == w.dst.block_size and n0 > 0:
        rb, bs = w.src.row_bytes, w.src.block_size
        want = torch.cat([hsrc[0][b * bs * rb:(b + 1) * bs * rb] for b in b0])[:n0 * rb]
        checked = bool(torch.equal(hdst[0][:n0 * rb], want))
        assert checked, "host-pool e2e result differs from the producer KV"
    return {"value": round(bytes_step / dt / 1e9, 2), "unit": "GB/s", "ms_per_step": round(dt * 1e3, 3),
            "steps": args.e2e_steps, "result_checked": checked,
            "h2d_bytes_per_step": bytes_step // 2, "d2h_bytes_per_step": bytes_step // 2,
            "how": "producer pool in pinned host memory, consumer pool on the device, staging pool in pinned host "
                   "memory: per layer kvx_push_layer_notify host -> device and kvx_push_layer (gather) device -> host, "
                   "both read or written over the chip-to-chip link by the copy kernel (the persistent plain-load "
                   "kernel, which the library runs for pools outside device memory); no separate copies; host wall "
                   "clock"}


def run_e2e(args, torch, kvx, w, src, dst, sp, dp, reqs, opts, bytes_step, world):
    """Producer KV from pinned host memory, per layer: H2D copy of the producer layer, push into the
    consumer pool, gather of the pushed consumer blocks (a second kvx plan, consumer -> a dense staging
    pool in request order) and D2H of that staging layer, on three streams so that copies in both
    directions overlap the pushes; plans built and synced each step. The result read back is exactly
    the pushed blocks; for equal layouts it must equal the producer blocks, which is checked."""
    L, P = w.src.n_layers, w.src.n_planes * w.src.n_shards
    bb_s = w.src.block_size * w.src.row_bytes
    s_lo = min(int(r[1][:-(-r[0] // w.src.block_size)].min()) for r in reqs if r[0] > 0)
    s_hi = max(int(r[1][:-(-r[0] // w.src.block_size)].max()) for r in reqs if r[0] > 0) + 1
    s_rng = (s_lo * bb_s, s_hi * bb_s)
    # staging: the requests' consumer blocks, densely, in request order
    nb = [-(-n // w.dst.block_size) for n, _, _ in reqs]
    off = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
    stage_geom = w.dst.replace(n_blocks=int(off[-1]))
    stage_reqs = [(n, d[:k], np.arange(off[i], off[i] + k, dtype=np.int32))
                  for i, ((n, _, d), k) in enumerate(zip(reqs, nb))]
    per = -(-stage_geom.buffer_bytes // 512) * 512
    stage_big = torch.empty(per * stage_geom.n_buffers, dtype=torch.uint8, device=src[0].device)
    stage = [stage_big[i * per:i * per + stage_geom.buffer_bytes] for i in range(stage_geom.n_buffers)]
    stp = kvx.Pool(stage_geom, stage)
    # one pinned allocation per side, cut into the buffers (16-byte aligned pieces)
    hs_n = -(-(s_rng[1] - s_rng[0]) // 4096) * 4096
    hd_n = -(-stage_geom.buffer_bytes // 4096) * 4096
    host_src_big = torch.empty(hs_n * len(src), dtype=torch.uint8, pin_memory=True)
    host_dst_big = torch.empty(hd_n * len(stage), dtype=torch.uint8, pin_memory=True)
    host_src = [host_src_big[i * hs_n:i * hs_n + (s_rng[1] - s_rng[0])] for i in range(len(src))]
    host_dst = [host_dst_big[i * hd_n:i * hd_n + stage_geom.buffer_bytes] for i in range(len(stage))]
    for h, d in zip(host_src, src):
        h.copy_(d[s_rng[0]:s_rng[1]])
    h2d, side, d2h = torch.cuda.Stream(), torch.cuda.Stream(priority=-1), torch.cuda.Stream()
    ev_h = [torch.cuda.Event() for _ in range(L)]
    ev_p = [torch.cuda.Event() for _ in range(L)]
    ev_g = [torch.cuda.Event() for _ in range(L)]
    ev_d = [torch.cuda.Event() for _ in range(L)]
    for ev in ev_h + ev_p + ev_g + ev_d:                # materialise the event handles
        ev.record(h2d)
    nd = stage_geom.n_planes * stage_geom.n_shards

    def issue():
        """One step, enqueued: per layer H2D -> push -> gather -> D2H. A layer's H2D waits for the
        previous step's D2H of that layer (which came after its push and gather), so consecutive steps
        pipeline layer by layer without overwriting a buffer still being read."""
        plan = kvx.kvx_plan_ex(sp, dp, reqs, opts)
        gather = kvx.kvx_plan_ex(dp, stp, stage_reqs, opts)
        for layer in range(L):
            with torch.cuda.stream(h2d):
                h2d.wait_event(ev_d[layer])
                for i in range(layer * P, (layer + 1) * P):
                    src[i][s_rng[0]:s_rng[1]].copy_(host_src[i], non_blocking=True)
                ev_h[layer].record(h2d)
            kvx.kvx_push_layer_notify(plan, layer, layer + 1, side, ev_h[layer], ev_p[layer])
            kvx.kvx_push_layer_notify(gather, layer, layer + 1, side, ev_p[layer], ev_g[layer])
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_g[layer])
                for i in range(layer * nd, (layer + 1) * nd):
                    host_dst[i].copy_(stage[i], non_blocking=True)
                ev_d[layer].record(d2h)
        return plan, gather

    def finish(plans):
        for pl in plans:
            assert kvx.kvx_sync(pl, -1) == kvx.KVX_OK
            kvx.kvx_plan_destroy(pl)

    done_at = []                                      # host time each step's plans were found complete

    def run(n):
        """n steps, each finished (plans synced) after the next one is enqueued."""
        prev = None
        for _ in range(n):
            cur = issue()
            if prev is not None:
                finish(prev)
                done_at.append(time.perf_counter())
            prev = cur
        finish(prev)
        d2h.synchronize()
        done_at.append(time.perf_counter())

    run(2)
    torch.cuda.synchronize()
    t = time.perf_counter()
    done_at.clear()
    run(args.e2e_steps)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t) / args.e2e_steps
    # interior intervals only: the first also holds the pipeline's fill, the last its drain
    step_ms = [(b - a) * 1e3 for a, b in zip(done_at[:-2], done_at[1:-1])] or [dt * 1e3]
    checked = None
    if w.src == w.dst.replace(n_blocks=w.src.n_blocks) and all(
            np.array_equal(np.asarray(r[1][:k]), np.arange(s_lo, s_lo + k)) for r, k in zip(reqs[:1], nb[:1])):
        # equal layouts, first request's producer blocks contiguous from s_lo: its gathered tokens must
        # equal those producer bytes, for the first and last buffer
        n0 = int(reqs[0][0]) * w.src.row_bytes if w.src.layout == kvx_inputs.LAYOUT_NHD else 0
        checked = all(torch.equal(host_dst[i][:n0], host_src[i][:n0]) for i in (0, len(host_dst) - 1))
        assert checked, "e2e result read back differs from the producer KV"
    return {"value": round(bytes_step / dt / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": sum(h.numel() for h in host_src),
            "d2h_bytes_per_step": sum(h.numel() for h in host_dst),
            "ms_per_step": round(dt * 1e3, 3), "steps": args.e2e_steps, "result_checked": checked,
            "step_ms": {"median": round(statistics.median(step_ms), 3), "min": round(min(step_ms), 3),
                        "max": round(max(step_ms), 3),
                        "how": "host time between consecutive steps found complete, the pipeline's fill and drain "
                               "left out; "
                               "the chip-to-chip link is shared with the host's other traffic, and runs saw "
                               "stretches of slower copies"},
            "how": "pinned host producer KV -> H2D per layer -> kvx_push_layer -> kvx gather of the pushed consumer "
                   "blocks into a dense staging pool -> D2H, 3 streams; a layer's H2D waits for the previous step's "
                   "D2H of that layer, each step's plans synced after the next step is enqueued; host wall clock "
                   "with device sync on both sides (rank 0)"}


def publish_turn(torch, kvx, w, hashes, d, turn_blocks):
    """Incremental publishing: each session's last `turn_blocks` full blocks (one turn's new tokens)
    hashed from the published hash of the block before them (kvx_block_hashes_ex), checked against
    the tail of the from-scratch chain. Returns (median ms over 4 timed calls, blocks hashed)."""
    bs = 64
    n_full = np.diff(w.rem_off)
    keep = np.minimum(n_full, turn_blocks)
    first = n_full - keep                                     # first new block of each session
    tok = [w.tokens[w.tok_off[s] + first[s] * bs: w.tok_off[s] + n_full[s] * bs] for s in range(w.n_sessions)]
    tok_off = np.concatenate([[0], np.cumsum([len(t) for t in tok])]).astype(np.int64)
    hash_off = np.concatenate([[0], np.cumsum(keep)]).astype(np.int64)
    host_hash = hashes.cpu().numpy().view(np.uint64)
    parent = np.array([host_hash[w.rem_off[s] + first[s] - 1] if first[s] > 0 else 0
                       for s in range(w.n_sessions)], dtype=np.uint64)
    want = np.concatenate([host_hash[w.rem_off[s] + first[s]: w.rem_off[s + 1]] for s in range(w.n_sessions)])
    toks, toff, hoff, par = d(np.concatenate(tok)), d(tok_off), d(hash_off), d(parent)
    out = torch.empty(max(int(hash_off[-1]), 1), dtype=torch.int64, device=hashes.device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    for _ in range(5):
        s.record()
        kvx.kvx_block_hashes_ex(toks, toff, w.n_sessions, bs, par, out, hoff)
        e.record()
        e.synchronize()
        ms.append(s.elapsed_time(e))
    got = out[:int(hash_off[-1])].cpu().numpy().view(np.uint64)
    if not np.array_equal(got, want):
        raise RuntimeError("incremental block hashes differ from the full chain's tail")
    return statistics.median(ms[1:]), int(hash_off[-1])


def run_match(torch, kvx, device, push_opts=None):
    """Prefix match of the bidirectional workload (256 sessions, 1024 shared + U[2k,32k] history tokens,
    block 64): decode publishes block hashes (kvx_block_hashes), prefill keeps a Bernoulli(0.4) subset
    in its table, kvx_match_prefix decides per session and builds the decode->prefill plan, which is
    then pushed for one layer of the fp8 576-byte latent pool."""
    w = kvx_inputs.bidir_mla_fp8(n_layers=1)

    def d(a):
        a = np.ascontiguousarray(a)
        view = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
        return torch.from_numpy(a.view(view)).to(device)

    tokens, tok_off, rem_off = d(w.tokens), d(w.tok_off), d(w.rem_off)
    n_pub = int(w.rem_off[-1])
    hashes = torch.empty(n_pub, dtype=torch.int64, device=device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hash_ms = []
    for _ in range(5):
        s.record()
        kvx.kvx_block_hashes(tokens, tok_off, w.n_sessions, 64, hashes, rem_off)
        e.record()
        e.synchronize()
        hash_ms.append(s.elapsed_time(e))
    turn_ms, turn_blocks = publish_turn(torch, kvx, w, hashes, d, turn_blocks=8)
    resident = torch.from_numpy(w.resident).to(device)
    keys = torch.unique(hashes[resident])
    table = kvx.kvx_table_build(keys, torch.arange(keys.numel(), dtype=torch.int32, device=device), keys.numel())
    out = torch.empty(w.n_sessions * 24, dtype=torch.uint8, device=device)
    rblk, free = d(w.remote_blk), d(w.free_blocks)
    src, _ = alloc_pool(torch, w.decode, "src", w.seed, device)
    dst, _ = alloc_pool(torch, w.prefill, "dst", 0, device)
    sp, dp = kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst)

    def match(with_plan):
        return kvx.kvx_match_prefix(tokens, tok_off, w.n_sessions, 64, table, hashes, rblk, rem_off, w.threshold,
                                    free, len(w.free_blocks), sp, dp, out, want_plan=with_plan)

    match_ms, plan_ms = [], []
    n_calls = 101                                     # the first of each kind is a warm-up
    for i in range(n_calls):
        t = time.perf_counter()
        _, plan = match(False)
        match_ms.append((time.perf_counter() - t) * 1e3)
    for i in range(n_calls):
        t = time.perf_counter()
        _, plan = match(True)
        plan_ms.append((time.perf_counter() - t) * 1e3)
        if i < n_calls - 1:
            kvx.kvx_plan_destroy(plan)
    res = out.cpu().numpy().view(kvx.MATCH_RESULT_DTYPE)
    # the hole-filling variant (resident blocks anywhere in the remote prefix are reused), decisions only
    out2 = torch.empty_like(out)
    holes_ms = []
    for i in range(n_calls):
        t = time.perf_counter()
        kvx.kvx_match_prefix(tokens, tok_off, w.n_sessions, 64, table, hashes, rblk, rem_off, w.threshold, free,
                             len(w.free_blocks), sp, dp, out2, want_plan=False, flags=kvx.KVX_MATCH_FILL_HOLES)
        holes_ms.append((time.perf_counter() - t) * 1e3)
    res_holes = out2.cpu().numpy().view(kvx.MATCH_RESULT_DTYPE)
    info = kvx.kvx_plan_get_info(plan)
    side = torch.cuda.Stream()
    kvx.kvx_plan_set_opts(plan, dict(push_opts or {}, flags=kvx.KVX_PLAN_TIMING))
    info = kvx.kvx_plan_get_info(plan)
    kvx.kvx_push_layer(plan, 0, side)
    kvx.kvx_sync(plan, -1)
    push_ms = []
    for _ in range(5):
        kvx.kvx_push_layer(plan, 0, side)
        kvx.kvx_sync(plan, -1)
        s_us, e_us = kvx.kvx_plan_push_times(plan)
        push_ms.append(float(e_us[0] - s_us[0]) * 1e-3)
    kvx.kvx_plan_destroy(plan)
    kvx.kvx_table_destroy(table)
    compares = int(res["remote_hit_blocks"].sum())
    m_ms = statistics.median(match_ms[1:])
    return {
        "workload": "bidir_mla_fp8: 256 sessions, block 64, threshold 512, fp8 latent 576 B, 1 of 48 layers pushed",
        "sessions_per_s": round(w.n_sessions / (m_ms * 1e-3), 1),
        "block_compares_per_s": round(compares / (m_ms * 1e-3), 1),
        "match_ms": round(m_ms, 3), "match_and_plan_ms": round(statistics.median(plan_ms[1:]), 3),
        "match_fill_holes_ms": round(statistics.median(holes_ms[1:]), 3),
        "fill_holes_push_blocks": int(res_holes["missing_tokens"].sum() // 64),
        "hash_only_ms": round(statistics.median(hash_ms[1:]), 3),
        "publish_turn_ms": round(turn_ms, 3), "publish_turn_blocks": turn_blocks,
        "hashed_blocks": n_pub, "pushing_sessions": int(res["push"].sum()),
        "push_blocks": int(res["missing_tokens"].sum() // 64), "runs": info["n_runs"],
        "dp_push_gbs_one_layer": round(2 * info["bytes_per_layer"] / (statistics.median(push_ms) * 1e-3) / 1e9, 1),
        "dp_push_kernel": KERNEL_SHORT[info["kernel"]], "dp_push_tile_bytes": info["tile_bytes"],
        "how": "host wall clock per kvx_match_prefix call (it waits for its stream), median of 100 calls; hashes and "
               "push with CUDA events",
    }


def bidir_full(torch, kvx, device, push_opts=None, reps=2, n_waves=4):
    """Configuration 5 whole: 256 sessions, all 48 layers of the fp8 576-byte latent pools (decode about
    130 GB, prefill about 87 GB), matched and pushed decode->prefill in waves of 64 sessions into one
    recycled free region, as a prefill instance would pull each turn's reusable spans. The decode side
    publishes its block hashes (kvx_block_hashes); the free region is sized by a decision-only pass
    (the largest wave's need). Per wave: kvx_match_prefix with its device-built plan (host wall clock;
    the call waits for its stream), then the 48 layer pushes on a side stream, their duration from
    the kernels' own global-timer stamps (first start to last end of the wave). `reps` timed rounds
    over all waves after one untimed round."""
    w0 = kvx_inputs.bidir_mla_fp8(n_layers=48, free_blocks=1)
    bs = w0.block_size

    def d(a):
        a = np.ascontiguousarray(a)
        view = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
        return torch.from_numpy(a.view(view)).to(device)

    tokens, tok_off, rem_off = d(w0.tokens), d(w0.tok_off), d(w0.rem_off)
    hashes = torch.empty(int(w0.rem_off[-1]), dtype=torch.int64, device=device)
    kvx.kvx_block_hashes(tokens, tok_off, w0.n_sessions, bs, hashes, rem_off)
    keys = torch.unique(hashes[torch.from_numpy(w0.resident).to(device)])
    table = kvx.kvx_table_build(keys, torch.arange(keys.numel(), dtype=torch.int32, device=device), keys.numel())
    per = w0.n_sessions // n_waves
    waves = []
    for k in range(n_waves):
        s0, s1 = k * per, (k + 1) * per
        t0, t1, r0, r1 = (int(x) for x in (w0.tok_off[s0], w0.tok_off[s1], w0.rem_off[s0], w0.rem_off[s1]))
        waves.append((tokens[t0:t1], d(w0.tok_off[s0:s1 + 1] - t0), hashes[r0:r1], d(w0.remote_blk[r0:r1]),
                      d(w0.rem_off[s0:s1 + 1] - r0)))
    out = torch.empty(per * 24, dtype=torch.uint8, device=device)
    dummy = torch.zeros(1, dtype=torch.int32, device=device)
    need = []
    for tk, to, hs, rb, ro in waves:                  # decisions only: how many blocks each wave pulls
        kvx.kvx_match_prefix(tk, to, per, bs, table, hs, rb, ro, w0.threshold, dummy, 0, None, None, out,
                             want_plan=False)
        res = out.cpu().numpy().view(kvx.MATCH_RESULT_DTYPE)
        need.append(int(res["missing_tokens"][res["push"] == 1].sum()) // bs)
    w = kvx_inputs.bidir_mla_fp8(n_layers=48, free_blocks=max(need))
    assert np.array_equal(w.remote_blk, w0.remote_blk) and np.array_equal(w.tokens, w0.tokens)
    src, _ = alloc_pool(torch, w.decode, "src", w.seed, device)
    dst, _ = alloc_pool(torch, w.prefill, "dst", 0, device)
    sp, dp = kvx.Pool(w.decode, src), kvx.Pool(w.prefill, dst)
    free = d(w.free_blocks)
    side = torch.cuda.Stream()
    match_ms, span_us, busy_us, launches, bytes_moved, blocks = [], [], [], 0, 0, 0
    for rep in range(reps + 1):
        for tk, to, hs, rb, ro in waves:
            t = time.perf_counter()
            st, plan = kvx.kvx_match_prefix(tk, to, per, bs, table, hs, rb, ro, w.threshold, free, len(w.free_blocks),
                                            sp, dp, out, want_plan=True)
            ms = (time.perf_counter() - t) * 1e3
            if st != kvx.KVX_OK:
                raise RuntimeError(f"kvx_match_prefix: {kvx.kvx_status_str(st)}")
            kvx.kvx_plan_set_opts(plan, dict(push_opts or {}, flags=kvx.KVX_PLAN_TIMING))
            info = kvx.kvx_plan_get_info(plan)
            for layer in range(48):
                kvx.kvx_push_layer(plan, layer, side)
            if kvx.kvx_sync(plan, -1) != kvx.KVX_OK:
                raise RuntimeError(f"kvx_sync: {kvx.kvx_last_error()}")
            s_ns, e_ns = kvx.kvx_plan_push_times_ns(plan)
            kvx.kvx_plan_destroy(plan)
            if rep == 0:
                continue
            base = s_ns.min()
            s_us, e_us = (s_ns - base) * 1e-3, (e_ns - base) * 1e-3
            match_ms.append(ms)
            span_us.append(float(e_us.max()))
            busy_us.append(union_us(s_us, e_us))
            launches += len(s_ns)
            bytes_moved += 2 * info["bytes_per_layer"] * 48
            res = out.cpu().numpy().view(kvx.MATCH_RESULT_DTYPE)
            blocks += int(res["missing_tokens"][res["push"] == 1].sum()) // bs
    kvx.kvx_table_destroy(table)
    peak, _ = measured_peak()
    span, busy = sum(span_us) * 1e-6, sum(busy_us) * 1e-6
    result = {"workload": "bidir_mla_fp8_full", "sessions": w.n_sessions, "layers": 48, "waves": n_waves,
              "timed_rounds": reps, "pull_blocks_per_round": blocks // reps, "wave_need_blocks": need,
              "bytes_per_round": bytes_moved // reps,
              "value": round(bytes_moved / span / 1e9, 2), "unit": "GB/s",
              "blocks_per_s": round(blocks / span, 1),
              "roofline_frac": round(bytes_moved / busy / 1e9 / peak, 4),
              "push_ms_per_round": round(span * 1e3 / reps, 3),
              "match_and_plan_ms_per_wave": round(statistics.median(match_ms), 3),
              "launches": launches, "kernel": KERNEL_NAMES[info["kernel"]], "threads": info["threads"],
              "how": "per round: 4 waves of 64 sessions, each kvx_match_prefix (decisions + device-built plan) "
                     "then 48 kvx_push_layer on a side stream into the recycled free region; GB/s = read+write "
                     "bytes / sum over waves of (last push end - first push start), kernel stamps; blocks/s = "
                     "pulled blocks (each all 48 layers) / the same time; roofline_frac over the union of the "
                     "push intervals"}
    del src, dst, sp, dp
    return result


# ---------------------------------------------------------------------------------------------
# oracle (CPU) timing: the cpu_baseline leg and the reference arm
# ---------------------------------------------------------------------------------------------

def oracle_sample(w, n_layers):
    """Host pools for `n_layers` layers of the workload (random bytes: the oracle copies opaque bytes)."""
    sg, dg = w.src.replace(n_layers=n_layers), w.dst.replace(n_layers=n_layers)
    rng = np.random.default_rng(w.seed)
    src = [rng.integers(0, 256, sg.buffer_bytes, dtype=np.uint8) for _ in range(sg.n_buffers)]
    dst = [np.full(dg.buffer_bytes, 0xAD, np.uint8) for _ in range(dg.n_buffers)]
    return sg, src, dg, dst


def oracle_layer(sg, src, dg, dst, layer):
    """One layer of the host sample as a one-layer pool pair (views, no copies)."""
    ps, pd = sg.n_planes * sg.n_shards, dg.n_planes * dg.n_shards
    return (sg.replace(n_layers=1), src[layer * ps:(layer + 1) * ps], dg.replace(n_layers=1),
            dst[layer * pd:(layer + 1) * pd])


def oracle_threads():
    """Host cores this process may run on (at most 32, which bounds the host sample's memory)."""
    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def cpu_baseline(w, seconds):
    """The oracle as it stands, on the host's cores: every thread pushes its own layer of a host
    sample of the workload, concurrently (the oracle's calls release the interpreter lock), for about
    `seconds`; then one thread alone, for comparison."""
    import concurrent.futures as cf
    import oracle
    orc = oracle.load()
    n_threads = oracle_threads()
    sg, src, dg, dst = oracle_sample(w, n_threads)
    reqs = requests(w)
    per_layer = 2 * sum(n for n, _, _ in reqs) * sg.n_shards * sg.row_bytes * sg.n_planes

    def loop(layer, deadline):
        views, n = oracle_layer(sg, src, dg, dst, layer), 0
        while True:
            orc.push(*views, reqs)
            n += 1
            if time.perf_counter() >= deadline:
                return n

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(n_threads) as pool:
        reps = sum(pool.map(lambda l: loop(l, t0 + 0.7 * seconds), range(n_threads)))
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    reps1 = loop(0, t1 + 0.3 * seconds)
    dt1 = time.perf_counter() - t1
    return {"value": round(per_layer * reps / dt / 1e9, 3), "unit": "GB/s", "cores": n_threads, "kind": "oracle",
            "sample": f"{reps} oracle pushes of one layer of {w.name} (host pools), {n_threads} threads each on "
                      f"its own layer, {dt:.1f} s",
            "single_thread": {"value": round(per_layer * reps1 / dt1 / 1e9, 3), "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} one-layer pushes, 1 thread, {dt1:.1f} s"}}


def oracle_push_rate(w, seconds, n_threads):
    """The oracle as it stands pushing one layer of workload `w` (host pools: the producer layer shared,
    one consumer copy per thread): all threads at once for 0.7 x `seconds`, then one thread for
    0.3 x `seconds`. GB/s counts read + write bytes; blocks/s counts producer blocks (block-layers)."""
    import concurrent.futures as cf
    import oracle
    orc = oracle.load()
    sg, dg = w.src.replace(n_layers=1), w.dst.replace(n_layers=1)
    rng = np.random.default_rng(w.seed)
    src = [rng.integers(0, 256, sg.buffer_bytes, dtype=np.uint8) for _ in range(sg.n_buffers)]
    dsts = [[np.full(dg.buffer_bytes, 0xAD, np.uint8) for _ in range(dg.n_buffers)] for _ in range(n_threads)]
    reqs = requests(w)
    per = 2 * sum(n for n, _, _ in reqs) * sg.n_shards * sg.row_bytes * sg.n_planes
    blocks = sum(-(-n // sg.block_size) for n, _, _ in reqs)

    def loop(dst, deadline):
        n = 0
        while True:
            orc.push(sg, src, dg, dst, reqs)
            n += 1
            if time.perf_counter() >= deadline:
                return n

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(n_threads) as pool:
        reps = sum(pool.map(lambda dst: loop(dst, t0 + 0.7 * seconds), dsts))
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    reps1 = loop(dsts[0], t1 + 0.3 * seconds)
    dt1 = time.perf_counter() - t1
    return {"workload": w.name, "value": round(per * reps / dt / 1e9, 3), "unit": "GB/s",
            "blocks_per_s": round(blocks * reps / dt, 1), "cores": n_threads, "kind": "oracle",
            "sample": f"{reps} oracle pushes of one layer ({per / 2e6:.1f} MB read), {n_threads} threads at once, "
                      f"{dt:.1f} s",
            "single_thread": {"value": round(per * reps1 / dt1 / 1e9, 3), "unit": "GB/s",
                              "blocks_per_s": round(blocks * reps1 / dt1, 1), "cores": 1,
                              "sample": f"{reps1} one-layer pushes, 1 thread, {dt1:.1f} s"}}


def oracle_bidir(seconds, n_threads):
    """The bidirectional workload on the oracle. Full scale (256 sessions): the match decision alone
    (oracle_match hashes every session's blocks and decides), one thread. Reduced (16 sessions, the
    same generator): end to end -- the published hashes, the match with its pairs, and the
    decode->prefill push of the pulled blocks -- with the push timed per layer (one thread, and all
    threads at once, one layer each) and the 48-layer figure composed from those times."""
    import concurrent.futures as cf
    import oracle
    orc = oracle.load()
    full = kvx_inputs.bidir_mla_fp8(n_layers=1)
    hs = np.concatenate([orc.block_hashes(full.tokens[full.tok_off[s]:full.tok_off[s + 1]], 64)
                         for s in range(full.n_sessions)])
    keys = np.unique(hs[full.resident])
    t = time.perf_counter()
    n_match = 0
    while True:
        m = orc.match(full.tokens, full.tok_off, 64, keys, hs, full.remote_blk, full.rem_off, full.threshold,
                      full.free_blocks)
        n_match += 1
        if time.perf_counter() - t >= 0.15 * seconds:
            break
    match_s = (time.perf_counter() - t) / n_match
    compares = int(m["remote_hit"].sum())

    w = kvx_inputs.bidir_mla_fp8(n_sessions=16, n_layers=1)
    t = time.perf_counter()
    hs16 = np.concatenate([orc.block_hashes(w.tokens[w.tok_off[s]:w.tok_off[s + 1]], 64) for s in range(w.n_sessions)])
    keys16 = np.unique(hs16[w.resident])
    m16 = orc.match(w.tokens, w.tok_off, 64, keys16, hs16, w.remote_blk, w.rem_off, w.threshold, w.free_blocks)
    hash_match_s = time.perf_counter() - t
    reqs, k = [], 0
    for s in range(w.n_sessions):
        if m16["push"][s]:
            nb = int(m16["missing"][s]) // 64
            reqs.append((nb * 64, m16["pair_src"][k:k + nb], m16["pair_dst"][k:k + nb]))
            k += nb
    pulled = k
    rng = np.random.default_rng(w.seed)
    src = [rng.integers(0, 255, w.decode.buffer_bytes, dtype=np.uint8)]
    dsts = [[np.full(w.prefill.buffer_bytes, kvx_inputs.CANARY_FP8, np.uint8)] for _ in range(n_threads)]
    per = 2 * pulled * 64 * 576

    def loop(dst, deadline):
        n = 0
        while True:
            orc.push(w.decode, src, w.prefill, dst, reqs)
            n += 1
            if time.perf_counter() >= deadline:
                return n

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(n_threads) as pool:
        reps = sum(pool.map(lambda dst: loop(dst, t0 + 0.5 * seconds), dsts))
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    reps1 = loop(dsts[0], t1 + 0.3 * seconds)
    dt1 = time.perf_counter() - t1
    layer_all, layer_one = dt / reps, dt1 / reps1          # seconds per layer: aggregate, one thread
    e2e_one = hash_match_s + 48 * layer_one
    e2e_all = hash_match_s + 48 * layer_all
    return {"workload": "bidir_mla_fp8", "kind": "oracle", "cores": n_threads,
            "match_full": {"sessions_per_s": round(full.n_sessions / match_s, 1),
                           "block_compares_per_s": round(compares / match_s, 1), "cores": 1,
                           "sample": f"{n_match} oracle_match calls on all 256 sessions ({len(hs)} published "
                                     f"blocks), 1 thread"},
            "e2e_16_sessions": {"sessions": w.n_sessions, "pulled_blocks": pulled,
                                "hash_and_match_ms": round(hash_match_s * 1e3, 3),
                                "push_gbs_one_layer": {"all_cores": round(per / layer_all / 1e9, 3),
                                                       "single_thread": round(per / layer_one / 1e9, 3)},
                                "blocks_per_s": {"all_cores": round(pulled / (48 * layer_all), 1),
                                                 "single_thread": round(pulled / (48 * layer_one), 1)},
                                "ms_48_layers": {"all_cores": round(e2e_all * 1e3, 1),
                                                 "single_thread": round(e2e_one * 1e3, 1)},
                                "sample": f"hashes + match once, then {reps} one-layer pushes on {n_threads} threads "
                                          f"({dt:.1f} s) and {reps1} on one ({dt1:.1f} s); 48-layer time = hash and "
                                          "match + 48 x the per-layer push time"}}


def cpu_baseline_per_config(seconds):
    """The oracle on each configuration beside the headline one, in the same run, each on all the
    host's cores and on one."""
    n = oracle_threads()
    out = []
    for name in ("tiny", "qwen3_32b_batched", "tp4_to_tp1_remap", "qwen3_32b_single_nhd_to_hnd"):
        out.append(oracle_push_rate(kvx_inputs.PUSH_WORKLOADS[name](n_layers=1) if name != "tiny"
                                    else kvx_inputs.tiny(), seconds, n))
        gc.collect()
    out.append(oracle_bidir(seconds, n))
    gc.collect()
    return out


def run_reference(args, rank, world):
    """The reference arm: the oracle (there is no other implementation of this path), each step one
    push of as many layers as the host has cores, one layer per thread, concurrently."""
    if rank != 0:
        return None
    import concurrent.futures as cf
    import oracle
    orc = oracle.load()
    w = kvx_inputs.PUSH_WORKLOADS[args.workload]()
    n_layers = n_threads = min(oracle_threads(), w.src.n_layers)
    sg, src, dg, dst = oracle_sample(w, n_layers)
    reqs = requests(w)
    bytes_step = 2 * sum(n for n, _, _ in reqs) * sg.n_shards * sg.row_bytes * sg.n_planes * n_layers
    views = [oracle_layer(sg, src, dg, dst, l) for l in range(n_layers)]
    # each thread runs the warm-up and then the timed steps of its own layer back to back; the K steps
    # are timed together, from a barrier after every warm-up to the last thread's end, so that no
    # step waits for the slowest thread of the one before
    start = threading.Barrier(n_threads + 1)

    def worker(v):
        for _ in range(args.warmup):
            orc.push(*v, reqs)
        start.wait()
        for _ in range(args.steps):
            orc.push(*v, reqs)

    with cf.ThreadPoolExecutor(n_threads) as pool:
        futs = [pool.submit(worker, v) for v in views]
        start.wait()
        t0 = time.perf_counter()
        for f in futs:
            f.result()
        dt = time.perf_counter() - t0
    v = round(bytes_step * args.steps / dt / 1e9, 3)
    sample = (f"each step: oracle push of {n_layers} of {w.src.n_layers} layers of {w.name} on host pools, "
              f"{n_threads} threads, one layer each; the steps run back to back per thread")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic: seeded random bytes, same block ids as the kvx arm",
            "config": {"workload": args.workload, "layers_per_step": n_layers},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": n_threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    # 32 hardware work queues for this process's streams (read by the CUDA runtime when it creates the
    # context, so set before any CUDA call; a caller's own setting wins). With the runtime's default of
    # 8, the bench's streams and the library's lanes share queues in an order that depends on when each
    # stream was created, and a lane that shares one with the prefill stream waits behind it: the same
    # push measured 0.88 or 0.97 of the copy peak on alternate calls in one process. The library sizes
    # its default lanes from the same variable.
    os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_kvx(args, rank, local_rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
