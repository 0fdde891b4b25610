#!/usr/bin/env python3
"""Benchmark of the MoE dispatch / combine hot path on GB300.

One step = ep_get_layout + ep_dispatch + ep_combine over one batch of
synthetic tokens (workloads.py).  Default workload: "grouped", the largest
single-GPU configuration (group-limited routing: T=16384 tokens, H=4096 bf16,
E=128 experts in 8 groups of 16, each token picks the top-4 groups by max
logit, then the top-8 experts in them; bf16 dispatch into the packed
expert-major buffer, weighted bf16 combine; 2.4 GB of algorithmic traffic per
step).  Small batches (decode: T=128, H=7168, E=256, top-8, fp8 into a
[256,128,7168] capacity buffer) run ep_layout_dispatch + ep_combine instead.

Metric: effective HBM GB/s of the step = algorithmic bytes (what the method
must move; see algorithmic_bytes) / device time, plus per-kernel us/call, GB/s
and fraction of the measured HBM copy bandwidth.

Timing: inputs resident in HBM.  The K timed steps run back to back in one
CUDA graph between two CUDA events, step i on set i % n of its own inputs and
outputs, with n sets whose data together is at least four times the 129 MB
L2, so every step's data is cold (inputs larger than L2).  The latency of one
step alone is also reported: one graph replay between two events after an L2
flush (a 512 MB write, then a 512 MB read, so the L2 holds only clean,
unrelated lines).  Per-kernel times
come from K more steps launched without a graph, with a CUDA event recorded
on the launching stream before and after every call; all of it is enqueued
behind the flush, so the calls run back to back as in the graph.  (Event
nodes inside a graph gave per-kernel times that grew by up to 2 us with the
number of graphs the process had instantiated, for the same kernel.)  Each
stage is also timed alone, after its own flush.  e2e: the same step through
the public API with pinned host inputs, host->device copies and the device->host
read of the combined output inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference   # the CPU oracle on the same workload

Multi-GPU: replicas (the single-GPU path has no exchange step); every rank
runs the full workload on its own GPU, value = all ranks' bytes / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import math
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

import workloads as W  # noqa: E402

METRIC = "dispatch/combine µs/call and effective HBM GB/s (1 GB300), % of HBM peak"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 * 10**6        # GB300 L2
MAX_SETS = 256
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ bytes

def algorithmic_bytes(wl: W.Workload, n_live: int) -> dict:
    """Bytes each kernel must move, counted once (no padding, no re-reads).

    layout:   read topk_idx, write slot_of, src_token/src_k for every receive
              row, counts/offsets/partition arrays.
    dispatch: read x once; write every live copy (bf16: H*2 bytes; fp8: H
              bytes + H/128 f32 scales).
    combine:  read every live row of y and topk_w / slot_of; write out.
    """
    T, H, k, E, P = wl.T, wl.H, wl.k, wl.E, wl.P
    N = T * k
    layout = 4 * N + 4 * N + 8 * wl.R + 4 * (2 * E + 2 * P + 2)
    if wl.fp8:
        dispatch = T * H * 2 + n_live * H + n_live * (H // 128) * 4
    else:
        dispatch = T * H * 2 + n_live * H * 2
    combine = n_live * H * 2 + T * H * 2 + T * k * (4 + 4)
    return dict(layout=layout, dispatch=dispatch, combine=combine)


def hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "layout": ("layout.cu",),
    "dispatch": ("dispatch.cu", "ring_schedule.h"),
    "layout_dispatch": ("layout_dispatch.cu",),
    "combine": ("combine.cu",),
}


def kernel_source_digest(kernel: str) -> str:
    """Digest of the sources a kernel is built from (its .cu plus the shared
    device header and launch declarations)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_ep_get_04_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + ("ep_device.cuh", "ep_kernels.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str) -> float | None:
    """DRAM bytes (read + write) per call of a kernel stage from the committed
    ncu summary profiles/traffic.txt, if it was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = kernel_source_digest(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split("#", 1)[0].split()
            if len(parts) == 4 and parts[0] == workload and parts[1] == kernel and parts[3] == digest:
                return float(parts[2])
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the benchmark runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), sm_max=float(parts[1]), power=float(parts[2]),
                                 hw=parts[4], hw_thermal=parts[5], sw_thermal=parts[6], sw_power=parts[7]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 0.25 * max(r2["power"] for r2 in rows)] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in busy), sm_max_mhz=max(r["sm_max"] for r in busy),
                    samples=len(busy), reasons=sorted(reasons))


# ------------------------------------------------------------- CPU oracle

def oracle_step(wl: W.Workload, inp: dict, y: np.ndarray):
    import oracle
    mode = oracle.CAPACITY if wl.mode == W.CAPACITY else oracle.PACKED
    L = oracle.layout(inp["topk_idx"], wl.E, wl.P, mode, wl.capacity)
    if wl.fp8:
        oracle.dispatch_fp8(inp["x"], L["slot_of"], wl.R)
    else:
        oracle.dispatch_bf16(inp["x"], L["slot_of"], wl.R)
    oracle.combine(y, inp["topk_w"], L["slot_of"])


def oracle_sample(wl: W.Workload, step_seconds: float = 1.0):
    """A bounded sample of the workload for the oracle: its first T' tokens,
    T' chosen so that one oracle step takes about step_seconds."""
    probe = wl.shrink(min(wl.T, 16))
    inp = W.make(probe)
    y = W.expert_rows(probe.R, probe.H)
    t0 = time.perf_counter()
    oracle_step(probe, inp, y)
    per_token = (time.perf_counter() - t0) / probe.T
    T_s = int(max(1, min(wl.T, step_seconds / max(per_token, 1e-9))))
    for _ in range(2):      # the 16-token probe misjudges the per-token cost: measure and rescale
        sample = wl.shrink(T_s) if T_s < wl.T else wl
        inp = W.make(sample)
        y = W.expert_rows(sample.R, sample.H)
        t0 = time.perf_counter()
        oracle_step(sample, inp, y)
        took = time.perf_counter() - t0
        T_new = int(max(1, min(wl.T, T_s * step_seconds / max(took, 1e-9))))
        if abs(T_new - T_s) <= 0.25 * T_s:
            break
        T_s = T_new
    n_live = int((inp["topk_idx"] >= 0).sum())
    return sample, inp, y, sum(algorithmic_bytes(sample, n_live).values())


def time_oracle(wl: W.Workload, budget_s: float = 12.0, min_reps: int = 3) -> dict:
    """The oracle, as it stands (single-threaded C), on a bounded sample."""
    sample, inp, y, total_bytes = oracle_sample(wl, step_seconds=min(1.0, budget_s / 4))
    times = []
    while len(times) < min_reps or sum(times) < budget_s:
        t0 = time.perf_counter()
        oracle_step(sample, inp, y)
        times.append(time.perf_counter() - t0)
    per_step = statistics.median(times)
    return dict(value=round(total_bytes / per_step / 1e9, 4), unit="GB/s", cores=1, kind="oracle",
                sample=f"first {sample.T} of {wl.T} tokens of the {wl.name} workload, whole "
                       f"layout+dispatch+combine step, {len(times)} steps, median {per_step * 1e3:.1f} ms/step, "
                       f"single-threaded C oracle",
                seconds=round(sum(times), 2), host_cpus=os.cpu_count())


# ------------------------------------------------------------- replicas

def max_over_ranks(vals: list[float], dist=None, device: str = "cpu") -> list[float]:
    """Element-wise max of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def percentiles_us(ms: list[float]) -> dict:
    """10th and 90th percentiles (µs) of per-call times given in ms."""
    if len(ms) < 2:
        return dict(us_p10=round(ms[0] * 1e3, 3), us_p90=round(ms[0] * 1e3, 3)) if ms else {}
    q = statistics.quantiles(ms, n=10, method="inclusive")
    return dict(us_p10=round(q[0] * 1e3, 3), us_p90=round(q[-1] * 1e3, 3))


def n_rotating_sets(step_bytes: int) -> int:
    """Independent input/output sets the timed steps rotate over: enough that
    their data together is at least four times the L2."""
    return max(1, min(MAX_SETS, math.ceil(4 * L2_BYTES / step_bytes)))


def workload_config(wl: W.Workload, step_bytes: int, world: int) -> dict:
    """The `config` object of the bench line; both arms print the same one."""
    n_sets = n_rotating_sets(step_bytes)
    return {"workload": wl.name, "description": wl.description, "T": wl.T, "H": wl.H, "E": wl.E,
            "top_k": wl.k, "partitions": wl.P, "layout": "capacity" if wl.mode == W.CAPACITY else "packed",
            "capacity": wl.capacity or None, "payload": "fp8_e4m3" if wl.fp8 else "bf16",
            "step_bytes": step_bytes,
            "l2": f"inputs larger than L2: the GPU arm's K timed steps rotate over {n_sets} independent sets of "
                  f"inputs and outputs ({n_sets} x {step_bytes / 1e6:.1f} MB touched, at least 4x the 129 MB L2), "
                  "L2 flushed once before the timed region; its per-kernel and latency figures flush before "
                  "every call.  The CPU oracle arm runs on the host",
            "parallelism": f"replicas x{world}"}


def replica_throughput(step_bytes: int, world: int, ms: float) -> float:
    """Whole-job GB/s of N replicas that each moved step_bytes in ms (max over ranks)."""
    return world * step_bytes / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------- GPU

def run_ours(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import combine_ep_get_04_gb300 as ep

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    wl = W.WORKLOADS[args.workload]
    inp = W.make(wl)
    cap = wl.capacity if wl.mode == W.CAPACITY else None
    plan = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, cap, fp8=wl.fp8)
    # The step's inputs live in one device buffer, [x | topk_idx | topk_w]
    # (x first: 16-byte aligned), so that the end-to-end run stages them with
    # one host-to-device copy per step.
    nx, ni = wl.T * wl.H * 2, wl.T * wl.k * 4
    stage_d = torch.empty(nx + 2 * ni, dtype=torch.uint8, device="cuda")
    x_d = stage_d[:nx].view(torch.bfloat16).view(wl.T, wl.H)
    idx_d = stage_d[nx:nx + ni].view(torch.int32).view(wl.T, wl.k)
    w_d = stage_d[nx + ni:].view(torch.float32).view(wl.T, wl.k)
    x_d.copy_(torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16))
    idx_d.copy_(torch.from_numpy(inp["topk_idx"]))
    w_d.copy_(torch.from_numpy(inp["topk_w"]))
    gen = torch.Generator(device="cuda").manual_seed(1234 + rank)
    y_d = torch.randn((plan.R, wl.H), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_src = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_dst = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush_l2():
        # Write a buffer 4x the L2, then read another one: the L2 ends up
        # holding only clean lines of unrelated data, so the timed kernels
        # neither hit their own data nor pay for earlier dirty lines.
        flush.zero_()
        torch.sum(flush_src, dim=0, keepdim=True, out=flush_dst)
    n_live = int((inp["topk_idx"] >= 0).sum())
    kbytes = algorithmic_bytes(wl, n_live)
    step_bytes = sum(kbytes.values())
    layout_launches = 2 if plan.workspace_bytes > 0 else 1

    def do_layout():
        plan.layout(idx_d, clear_flags=False)

    def do_dispatch():
        plan.dispatch(x_d)

    def do_layout_dispatch():
        plan.layout_dispatch(idx_d, x_d, clear_flags=False)

    def do_combine():
        plan.combine(y_d, w_d)

    # The step: ep_layout_dispatch (one launch for small batches) + ep_combine;
    # larger batches run the three calls that ep_layout_dispatch would make.
    fused = ep.fused_layout_dispatch(wl.T, wl.k, wl.E)
    if fused:
        stages = [("layout_dispatch", do_layout_dispatch, kbytes["layout"] + kbytes["dispatch"], 1),
                  ("combine", do_combine, kbytes["combine"], 1)]
    else:
        stages = [("layout", do_layout, kbytes["layout"], layout_launches),
                  ("dispatch", do_dispatch, kbytes["dispatch"], 1),
                  ("combine", do_combine, kbytes["combine"], 1)]
    names = tuple(n for n, _, _, _ in stages)
    nbytes = {n: b for n, _, b, _ in stages}
    launches_per_step = sum(c for _, _, _, c in stages)

    def do_step():
        for _, fn, _, _ in stages:
            fn()

    plan.layout_out.err_flags.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            do_step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    # Each stage alone after an L2 flush per call is the per-call figure of
    # the method's measurement plan; the variant ep_combine_src (combine
    # through the expert-side source maps, per-row weights) is timed the same
    # way.
    row_w_d = torch.rand(plan.R, generator=gen, device="cuda", dtype=torch.float32)

    def do_combine_src():
        plan.combine_src(y_d, row_w_d)

    alone_fns = [(n, fn) for n, fn, _, _ in stages] + [("combine_src", do_combine_src)]
    if wl.fp8:
        # combine over fp8 expert outputs: the dispatched codes and scales
        # themselves stand for the experts' outputs (ep_combine_fp8)
        def do_combine_fp8():
            plan.combine_fp8(plan.recv, plan.recv_scales, w_d)

        alone_fns.append(("combine_fp8", do_combine_fp8))
    graphs = {"step": capture(do_step)}
    if args.profile:
        # Only the step kernels, on one set of inputs (for ncu launch lists and
        # captures, with little device memory): W + K graph replays, each
        # behind an L2 flush; with --profile-variant, each followed by one
        # call of that variant behind its own flush.
        variant = dict(alone_fns).get(args.profile_variant) if args.profile_variant else None
        if args.profile_variant and variant is None:
            raise SystemExit(f"--profile-variant {args.profile_variant}: not run on the {wl.name} workload")
        for _ in range(args.warmup + args.steps):
            flush_l2()
            graphs["step"].replay()
            if variant is not None:
                flush_l2()
                variant()
        torch.cuda.synchronize()
        flags = int(plan.layout_out.err_flags.item())
        if rank == 0:
            print(json.dumps({"profile_run": wl.name, "steps": args.warmup + args.steps,
                              "launches_per_step": launches_per_step, "variant": args.profile_variant,
                              "err_flags": flags}))
        if dist is not None:
            dist.destroy_process_group()
        return None


    # ---- the timed region: K steps back to back in one graph, step i on set
    # i % n_sets of its own inputs and outputs, with enough sets that their
    # data together is at least four times the L2, so every step's data is
    # cold (inputs larger than L2 instead of a flush between steps).
    n_sets = n_rotating_sets(step_bytes)
    sets = [(plan, x_d, idx_d, w_d, y_d)]
    for _ in range(1, n_sets):
        p2 = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, cap, fp8=wl.fp8)
        st2 = stage_d.clone()
        sets.append((p2, st2[:nx].view(torch.bfloat16).view(wl.T, wl.H),
                     st2[nx:nx + ni].view(torch.int32).view(wl.T, wl.k),
                     st2[nx + ni:].view(torch.float32).view(wl.T, wl.k),
                     torch.randn((plan.R, wl.H), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)))

    def run_set(q):
        p2, x2, i2, w2, y2 = sets[q]
        if fused:
            p2.layout_dispatch(i2, x2, clear_flags=False)
        else:
            p2.layout(i2, clear_flags=False)
            p2.dispatch(x2)
        p2.combine(y2, w2)

    side.wait_stream(torch.cuda.current_stream())   # the sets' buffers were filled on this stream
    with torch.cuda.stream(side):
        for q in range(n_sets):
            run_set(q)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graphs["timed"] = capture(lambda: [run_set(q % n_sets) for q in range(args.steps)])

    # Each stage K times back to back over the same sets: the average launch
    # duration (total / K between two events), free of the per-launch rounding
    # of event times (completion reaches the events in steps of ~2 us here).
    def stage_call(n, q):
        p2, x2, i2, w2, y2 = sets[q]
        if n == "layout":
            p2.layout(i2, clear_flags=False)
        elif n == "dispatch":
            p2.dispatch(x2)
        elif n == "layout_dispatch":
            p2.layout_dispatch(i2, x2, clear_flags=False)
        elif n == "combine":
            p2.combine(y2, w2)
        elif n == "combine_src":
            p2.combine_src(y2, row_w_d)
        else:   # combine_fp8: the set's dispatched codes and scales stand for the expert outputs
            p2.combine_fp8(p2.recv, p2.recv_scales, w2)

    variants = ("combine_src", "combine_fp8") if wl.fp8 else ("combine_src",)
    for n in variants:          # one eager call each before capture
        stage_call(n, 0)
    torch.cuda.synchronize()
    for n in names + variants:
        graphs["b2b_" + n] = capture(lambda n=n: [stage_call(n, q % n_sets) for q in range(args.steps)])
    graphs["warm"] = capture(lambda: [run_set(q % n_sets) for q in range(args.warmup)])
    stream = torch.cuda.current_stream()

    def timed(g, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush_l2()
            a.record(stream)
            g.replay()
            b.record(stream)
        return evs

    sampler = ClockSampler(local_rank)
    sampler.start()
    # bring the clocks up (~0.5 s of back-to-back steps), then the warm-up steps
    t_end = time.perf_counter() + 0.5
    while time.perf_counter() < t_end:
        for _ in range(20):
            graphs["step"].replay()
        torch.cuda.synchronize()
    flush_l2()
    graphs["warm"].replay()                      # W warm-up steps
    flush_l2()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps, back to back, one pair of events
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record(stream)
    graphs["timed"].replay()
    ev_b.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    timed_ms = ev_a.elapsed_time(ev_b)

    # ---- latency of one step alone: K more steps, each one graph replay
    # between two events after its own L2 flush
    step_evs = timed(graphs["step"], args.steps)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_evs]

    # ---- per-kernel times, same flush discipline, K more steps: the calls of
    # a step launched one by one with an event on the stream between them,
    # all enqueued behind the flush so that they run back to back.
    kernel_ms = {n: [] for n in names}
    for _ in range(args.steps):
        flush_l2()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
        for q, (_, fn, _, _) in enumerate(stages):
            evs[q].record(stream)
            fn()
        evs[-1].record(stream)
        torch.cuda.synchronize()
        for q, n in enumerate(names):
            kernel_ms[n].append(evs[q].elapsed_time(evs[q + 1]))
    b2b_us = {}
    for n in names + variants:
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graphs["b2b_" + n].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        b2b_us[n] = e0.elapsed_time(e1) * 1e3 / args.steps
    alone_ms = {n: [] for n, _ in alone_fns}
    for n, fn in alone_fns:
        for _ in range(args.steps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            alone_ms[n].append(a.elapsed_time(b))
    per_kernel = {n: dict(us=round(statistics.median(kernel_ms[n]) * 1e3, 3),
                          us_mean=round(statistics.fmean(kernel_ms[n]) * 1e3, 3),
                          **percentiles_us(kernel_ms[n]),
                          timed="inside a step launched call by call, events on the stream between the calls")
                  for n in names}

    # ---- e2e through the public API with host buffers: every step copies its
    # inputs in from pinned host memory and the combined output back out.
    stage_h = torch.empty(nx + 2 * ni, dtype=torch.uint8).pin_memory()
    stage_h[:nx].view(torch.int16).copy_(torch.from_numpy(inp["x"].view(np.int16)).reshape(-1))
    stage_h[nx:nx + ni].view(torch.int32).copy_(torch.from_numpy(inp["topk_idx"]).reshape(-1))
    stage_h[nx + ni:].view(torch.float32).copy_(torch.from_numpy(inp["topk_w"]).reshape(-1))
    out_h = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    h2d = stage_h.numel()
    d2h = out_h.numel() * 2

    def do_e2e():
        stage_d.copy_(stage_h, non_blocking=True)   # x, topk_idx and topk_w in one copy
        do_step()
        out_h.copy_(plan.out, non_blocking=True)

    def time_e2e(run):
        evs = []
        for it in range(args.warmup + args.steps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            if it >= args.warmup:
                evs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    e2e_ms = time_e2e(do_e2e)                     # copies + the calls issued from Python
    g_e2e = capture(do_e2e)                       # the same, captured once as one graph
    e2e_graph_ms = time_e2e(g_e2e.replay)

    # Pipelined: the same per-step copies and calls, with the host->device
    # copy of step i+1 and the device->host copy of step i-1 overlapping step
    # i on their own streams (two device buffer sets, events guarding reuse).
    plan_b = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, cap, fp8=wl.fp8)
    stage_b = torch.empty_like(stage_d)
    out_hb = torch.empty_like(out_h).pin_memory()
    pipe_sets = [(plan, stage_d, out_h), (plan_b, stage_b, out_hb)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipe_step(i):
        p2, st, oh = pipe_sets[i % 2]
        b = i % 2
        if i >= 2:
            s_in.wait_event(ev_comp[b])           # step i-2 has read this input buffer
        with torch.cuda.stream(s_in):
            st.copy_(stage_h, non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        if i >= 2:
            s_comp.wait_event(ev_out[b])          # step i-2's output has been read back
        with torch.cuda.stream(s_comp):
            xs = st[:nx].view(torch.bfloat16).view(wl.T, wl.H)
            ids = st[nx:nx + ni].view(torch.int32).view(wl.T, wl.k)
            ws = st[nx + ni:].view(torch.float32).view(wl.T, wl.k)
            if fused:
                p2.layout_dispatch(ids, xs, clear_flags=False)
            else:
                p2.layout(ids, clear_flags=False)
                p2.dispatch(xs)
            p2.combine(y_d, ws)
            ev_comp[b].record(s_comp)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            oh.copy_(p2.out, non_blocking=True)
            ev_out[b].record(s_out)

    def pipe_run(n):
        # fork from the current stream, n pipelined steps, join back
        main = torch.cuda.current_stream()
        for s_ in (s_in, s_comp, s_out):
            s_.wait_stream(main)
        for i in range(n):
            pipe_step(i)
        for s_ in (s_in, s_comp, s_out):
            main.wait_stream(s_)

    pipe_run(args.warmup)                         # eager warm-up
    torch.cuda.synchronize()
    # The K pipelined steps captured as one CUDA graph (so that issuing from
    # Python does not pace small steps), replayed once between two events.
    g_pipe = torch.cuda.CUDAGraph()
    cap_s = torch.cuda.Stream()
    cap_s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g_pipe, stream=cap_s):
        pipe_run(args.steps)
    torch.cuda.synchronize()
    g_pipe.replay()                               # one untimed replay
    torch.cuda.synchronize()
    pe_a, pe_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe_a.record(stream)
    g_pipe.replay()
    pe_b.record(stream)
    torch.cuda.synchronize()
    e2e_pipe_ms = [pe_a.elapsed_time(pe_b) / args.steps]
    clocks = sampler.stop()

    flags = int(plan.layout_out.err_flags.item()) | int(plan_b.layout_out.err_flags.item())
    for p2, _, _, _, _ in sets[1:]:
        flags |= int(p2.layout_out.err_flags.item())
    if flags:
        raise RuntimeError(f"device error flags set during the benchmark: {flags:#x}")
    ms_mean = timed_ms / args.steps
    lat_mean = statistics.fmean(step_ms)
    e2e_mean = statistics.fmean(e2e_ms)
    e2e_graph_mean = statistics.fmean(e2e_graph_ms)
    e2e_pipe_mean = e2e_pipe_ms[0]
    ms_mean, lat_mean, e2e_mean, e2e_graph_mean, e2e_pipe_mean, wall = max_over_ranks(
        [ms_mean, lat_mean, e2e_mean, e2e_graph_mean, e2e_pipe_mean, wall], dist, "cuda")
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return None

    peak, peak_kind = hbm_peak()
    for name, r in per_kernel.items():
        gbs = nbytes[name] / (r["us"] * 1e-6) / 1e9
        r.update(bytes=nbytes[name], gbs=round(gbs, 1), frac_of_hbm=round(gbs / peak, 4))
    # combine through the source maps reads each live row's (token, position,
    # weight) record instead of the token-side slot and weight
    nbytes_alone = dict(nbytes, combine_src=kbytes["combine"] - 8 * wl.T * wl.k + 12 * n_live,
                        combine_fp8=n_live * wl.H + n_live * (wl.H // 128) * 4 + wl.T * wl.H * 2 + wl.T * wl.k * 8)
    alone = {}
    for name, ms in alone_ms.items():
        a_us = statistics.median(ms) * 1e3
        a_gbs = nbytes_alone[name] / (a_us * 1e-6) / 1e9
        alone[name] = dict(us=round(a_us, 3), **percentiles_us(ms), bytes=nbytes_alone[name], gbs=round(a_gbs, 1),
                           frac_of_hbm=round(a_gbs / peak, 4))
    b2b, b2b_var = {}, {}
    for name, us in b2b_us.items():
        gbs = nbytes_alone[name] / (us * 1e-6) / 1e9
        (b2b if name in names else b2b_var)[name] = dict(us=round(us, 3), gbs=round(gbs, 1),
                                                        frac_of_hbm=round(gbs / peak, 4))
    dominant = max(names, key=lambda n: b2b_us[n])
    ach = nbytes[dominant] / (b2b_us[dominant] * 1e-6) / 1e9
    traffic = ncu_traffic(wl.name, dominant)
    value = replica_throughput(step_bytes, world, ms_mean)
    e2e_value = replica_throughput(step_bytes, world, e2e_pipe_mean)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_mean, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8-e4m3+bf16" if wl.fp8 else "bf16", "data": "synthetic",
        "config": workload_config(wl, step_bytes, world),
        "method": {"timing": "the K steps in one CUDA graph between two CUDA events on the launching stream",
                   "calls": "ep_layout_dispatch + ep_combine" if fused else "ep_get_layout + ep_dispatch + ep_combine"},
        "latency": {"ms_per_step": round(lat_mean, 5),
                    "how": "one step per CUDA-graph replay between two CUDA events, L2 flushed before each, "
                           "mean of K"},
        "kernels": dict(per_kernel, resolution="completion of a kernel reaches CUDA events in steps of about "
                                               "2 us on this GPU, so a per-call figure under ~20 us is bound by "
                                               "that resolution, not by the kernel; kernels_back_to_back holds "
                                               "the average launch durations"),
        "kernels_alone": dict(alone, how="each stage launched alone between two CUDA events on the stream, "
                                          "L2 flushed before every call, median of K calls"),
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(ach / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": nbytes[dominant], "peak_source": f"{peak_kind} hbm_gbs",
                     "duration": "average launch duration: the kernel's stage K times back to back over the "
                                 "rotating sets in one CUDA graph, total / K between two CUDA events"},
        "kernels_back_to_back": dict(b2b, how="each stage K times back to back over the rotating sets (every "
                                              "launch on cold data), one CUDA graph, total / K between two events"),
        "variants_back_to_back": dict(b2b_var, how="the same for ep_combine_src (combine through the expert-side "
                                                   "source maps and per-row weights) and, for fp8 workloads, "
                                                   "ep_combine_fp8 over the dispatched codes and scales"),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_pipe_mean, 5),
                "how": "every step: x, topk_idx and topk_w from one pinned host buffer -> device in one copy, "
                       "the public-API calls, out -> pinned host; K steps pipelined over two device buffer sets "
                       "(the copy in of step i+1 and the copy out of step i-1 on their own streams overlap step "
                       "i), captured as one CUDA graph and timed from the first copy in to the last copy out",
                "serial": {"value": round(replica_throughput(step_bytes, world, e2e_mean), 2),
                           "ms_per_step": round(e2e_mean, 5),
                           "how": "the same step with its two copies, one step at a time (L2 flushed before "
                                  "each), issued from Python"},
                "graph": {"value": round(replica_throughput(step_bytes, world, e2e_graph_mean), 2),
                          "ms_per_step": round(e2e_graph_mean, 5),
                          "how": "the serial step captured once as one CUDA graph, replayed per step"}},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(wall, 4),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = time_oracle(wl, budget_s=args.cpu_seconds)
    return line


def run_reference(args, rank: int, world: int) -> dict | None:
    """The reference arm: the CPU oracle on the same workload, each step a
    bounded sample (rank 0 only; other ranks exit without work)."""
    if rank != 0:
        return None
    wl = W.WORKLOADS[args.workload]
    full = W.make(wl)
    step_bytes = sum(algorithmic_bytes(wl, int((full["topk_idx"] >= 0).sum())).values())
    del full
    step_s = min(1.0, max(0.05, args.cpu_seconds * 5 / max(1, args.steps + args.warmup)))
    sample, inp, y, total_bytes = oracle_sample(wl, step_seconds=step_s)
    times = []
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_step(sample, inp, y)
        if it >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = statistics.fmean(times)
    value = total_bytes / per_step / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3+bf16" if wl.fp8 else "bf16", "data": "synthetic",
        "config": dict(workload_config(wl, step_bytes, world), sample_tokens=sample.T),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {sample.T} of {wl.T} tokens of the {wl.name} workload per step, "
                                   f"single-threaded C oracle", "host_cpus": os.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(W.WORKLOADS), default="grouped")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-variant", choices=("combine_src", "combine_fp8"), default=None,
                    help="with --profile: also run this variant once after every step")
    ap.add_argument("--profile", action="store_true",
                    help="run only W+K flushed step replays (for an ncu launch list); prints no bench line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("for --gpus > 1 launch with torch.distributed.run (one rank per GPU)")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
