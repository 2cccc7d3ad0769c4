#!/usr/bin/env python
"""Benchmark of the Gated DeltaNet speculative verify/commit path on one GB300.

Metric: microseconds per layer-call (verify + commit of one layer) and the
achieved HBM GB/s of that layer-call, from the algorithmic bytes the method
must move (each checkpoint read, the tokens' q/k/v/gates, the outputs, the
committed states).

Workload (default): batch 64, 32 heads, dk = dv = 128, 16 draft tokens per
request, 24 independent layers called back to back, each request's state in a
24 x 512-slot fp32 pool (24 GiB), accepted lengths ~ Binomial(16, 0.75).  One
step = for every layer: gdn_verify then gdn_commit.  Every step touches about
11 GB, far more than the 129 MB L2, so no flush is needed between steps.  The
timed steps replay the step's calls captured once in a CUDA graph, as an
engine runs its decode step (--no-graph: launched one by one); the one-by-one
figure is measured and reported beside it either way.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (the slow reference this path is checked against).  Under torchrun
(N > 1) every rank runs its own replica of the workload (weak scaling; no data
is exchanged); the step time is the maximum over ranks, and `value` is the
whole job's microseconds per layer-call: that time over the layer-calls of all
ranks (so it falls as N grows).  The HBM fractions are then taken against N
GPUs' peak; the roofline entry stays the dominant kernel on one GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decode_gated_gb300 import inputs  # noqa: E402

WORKLOAD = "b64_h32_d128_t16_x24"
METRIC = "us per layer-call (verify+commit) and achieved HBM GB/s vs ~8 TB/s, 1xGB300"
UNIT = "us/layer-call"
NOMINAL_HBM_GBS = 8000.0
MODE_NAME = {"v": "verify", "c": "commit", "f": "fused", "cv": "commit_verify",
             "C": "commit_layers", "F": "fused_layers",  # upper case: one launch, all layers
             "a": "accept", "rv": "replay_verify", "rc": "replay_commit"}


# ----------------------------------------------------------------- accounting

def alg_bytes(prob, mode: str, o_bytes: int = 4) -> int:
    """Minimum bytes the method moves for one call, per unit (request, head):
    verify  = state read + T (q, k, v, alpha, beta) + T o
    commit  = [a > 0] (state read + state write) + a (k, v, alpha, beta)
    fused   = state read + [a > 0] state write + T (q, k, v, alpha, beta, o)
    plus per-request metadata (slot id, accepted length, sequence offsets)."""
    esz = 2 if prob.qkv_dtype == "bf16" else 4
    tile = prob.dk * prob.dv * 4
    q_k = prob.dk * esz
    v_ = prob.dv * esz
    o_ = prob.dv * o_bytes
    lens = prob.lengths.astype(np.int64)
    acc = prob.accepted.astype(np.int64)
    H = prob.heads
    meta = prob.batch * (4 + (4 if mode != "verify" else 0) + (4 if prob.ragged else 0))
    if mode == "verify":
        per_r = tile + lens * (2 * q_k + v_ + 8 + o_)
    elif mode == "commit":
        per_r = (acc > 0) * (2 * tile) + acc * (q_k + v_ + 8)
    elif mode == "commit_verify":
        # the previous step (here: the same problem one step earlier) commits its
        # accepted rows from its cached W: k, alpha and W of a rows; this step
        # verifies its drafts and caches their W (o-sized)
        meta += prob.batch * 4 * (2 if prob.ragged else 1)
        per_r = (tile + (acc > 0) * tile + acc * (q_k + 4 + o_)
                 + lens * (2 * q_k + v_ + 8 + o_ + o_))
    else:
        per_r = tile + (acc > 0) * tile + lens * (2 * q_k + v_ + 8 + o_)
    return int(H * per_r.sum() + meta)


def replay_bytes(prob, buf, mode: str) -> int:
    """Minimum bytes of one ReplaySSM call, per unit, with n = the slot's buffered rows:
    verify = state read + (n + T) buffered rows (k, v, alpha, beta) + T (q, o)
    commit = for a flushed slot (keep + max_T > C, keep = n + a): state read +
             state write + keep buffered rows; nothing else moves (pointer move)
    plus per-request metadata (slot id, buffered length, accepted length, new length)."""
    esz = 2 if prob.qkv_dtype == "bf16" else 4
    tile = prob.dk * prob.dv * 4
    row = prob.dk * esz + prob.dv * esz + 8  # one buffered row: k, v, alpha, beta
    lens = prob.lengths.astype(np.int64)
    n = np.array([int(buf["len_in"][int(s)]) for s in prob.slot_ids], dtype=np.int64)
    if mode == "verify":
        per_r = tile + (n + lens) * row + lens * (prob.dk * esz + prob.dv * 4)
        meta = prob.batch * 8
    else:
        keep = n + prob.accepted.astype(np.int64)
        flush = keep + int(prob.max_T) > int(buf["capacity"])
        per_r = flush * (2 * tile + keep * row)
        meta = prob.batch * 16
    return int(prob.heads * per_r.sum() + meta)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in rows:
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
                power.append(float(row[3]))
            except ValueError:
                continue
            for name, flag in zip(names, row[5:9]):
                if flag.strip().lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profile_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, if the
    kernel source has not changed since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.]+)", text)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_f = re.search(r"source_file:\s*(\S+)", text)
    if not (m_b and m_h and m_f):
        return None
    src = os.path.join(ROOT, m_f.group(1))
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m_h.group(1):
        return None
    return float(m_b.group(1))


def cpu_oracle_time(prob, n_units: int, threads: int):
    """Seconds the float64 oracle takes for verify + commit of n_units sampled
    units of one layer, and the per-layer-call extrapolation in microseconds."""
    import dataclasses

    import oracle

    # float64 copies up front, so the timed region holds the recurrence only
    p64 = dataclasses.replace(prob, **{f: np.asarray(getattr(prob, f), np.float64)
                                       for f in ("q", "k", "v", "alpha", "beta", "s0")})
    rng = np.random.default_rng(7)
    units = np.sort(rng.choice(prob.units, size=min(n_units, prob.units), replace=False))
    oracle.load()
    t0 = time.perf_counter()
    oracle.run_units(p64, units, want_o=True, want_state=False, threads=threads)
    oracle.run_units(p64, units, want_o=False, want_state=True, threads=threads)
    dt = time.perf_counter() - t0
    return dt, dt / len(units) * prob.units * 1e6, len(units)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer_call(ms_total: float, steps: int, layers: int, world: int) -> float:
    """The whole job's microseconds per layer-call: the slowest rank's time for
    `steps` steps, over the layer-calls of all `world` ranks (each rank runs
    `layers` layer-calls per step on its own replica)."""
    return ms_total * 1e3 / (steps * layers * world)


# ----------------------------------------------------------------- arms

def run_reference(args, rank):
    """The oracle on the host cores.  A step is one bounded sample: verify and
    commit passes over `--ref-units` units of layer 0.  `ms_per_step` is the wall
    time of that sample as it ran; `value` scales it to a whole layer-call
    (units of a layer-call / units of the sample)."""
    if rank != 0:
        return
    prob = inputs.make_problem(args.workload, layer=0)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        cpu_oracle_time(prob, args.ref_units, threads)
    times, walls = [], []
    n = 0
    for _ in range(args.steps):
        dt, us, n = cpu_oracle_time(prob, args.ref_units, threads)
        times.append(us)
        walls.append(dt)
    value = statistics.median(times)
    scale = prob.units / n
    sample = (f"{n} of {prob.units} units of layer 0 per step (verify pass + commit pass), "
              f"{statistics.median(walls):.2f} s wall per step, scaled by {scale:g} "
              f"to a full layer-call")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.fmean(walls) * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "order": "verify then commit per layer",
                   "step": f"{n} sampled units (ms_per_step is their wall time)",
                   "value_scale": scale},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- timing

def graph_of(calls, stream, reps=1):
    """`reps` steps' calls captured in one CUDA graph (the library's per-device
    set-up has run in the warm-up); returns a callable that replays it on
    `stream`."""
    import torch

    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    # thread-local capture: other threads of the process (NCCL's watchdog under
    # torchrun) may keep querying their own events meanwhile
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for _ in range(reps):
            for _, call in calls:
                call()
    torch.cuda.synchronize()

    def replay():
        g.replay()
    replay.keep = g
    return replay


def time_calls(calls, kinds, stream, steps, warmup, world, dev, check=(), graph=True):
    """Warm up, then timed regions of `steps` steps each (a step issues every
    call of `calls` once, in order, on `stream`):
      1. one event pair around all steps, launches back to back as in use (the
         headline figure): with `graph`, the steps are replays of a CUDA graph
         captured once, as an engine runs its decode step (a graph holds
         enough steps for at least 24 launches, so the gap between two
         replays is spread over them);
      1b. with `graph`, the same with the calls launched one by one;
      2. an event pair around every launch, for the per-kernel durations.
    Returns the slowest rank's region-1 milliseconds, the mean milliseconds of
    each call kind in region 2, the calls of each kind per step, and the
    region-1b milliseconds (None without `graph`)."""
    import torch
    import torch.distributed as dist

    from speculative_decode_gated_gb300 import binding

    def barrier():
        if world > 1:
            dist.barrier()

    def step(events=None):
        if events is None:
            for _, call in calls:
                call()
            return
        for m, call in calls:
            a, b = events[m][events["i"][m]]
            a.record(stream)
            call()
            b.record(stream)
            events["i"][m] += 1

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    for d in check:
        if binding.gdn_read_device_error(d.c) != 0:
            raise RuntimeError("device-side argument error during warm-up")
    region1, reps = step, 1
    if graph:
        reps = -(-24 // len(calls))  # steps per replay
        with torch.cuda.stream(stream):
            region1 = graph_of(calls, stream, reps)
            region1()
        torch.cuda.synchronize()
    runs = -(-steps // reps)  # region-1 iterations; steps_run = runs * reps
    n_per_step = {m: sum(1 for mm, _ in calls if mm == m) for m in kinds}
    events = {m: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n_per_step[m] * steps)] for m in kinds}
    events["i"] = {m: 0 for m in kinds}
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(runs):
        region1()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    # the time of `steps` steps at the measured rate (runs * reps steps ran)
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, dev) * steps / (runs * reps)
    ms_direct = None
    if graph:
        t_start.record(stream)
        for _ in range(steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_direct = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    for _ in range(steps):
        step(events)
    torch.cuda.synchronize()
    barrier()
    avg_ms = {m: statistics.fmean(a.elapsed_time(b) for a, b in events[m]) for m in kinds}
    return ms_total, avg_ms, n_per_step, ms_direct


def time_back_to_back(calls, kinds, stream, steps, world, dev):
    """Mean milliseconds per launch of each call kind when the step's launches
    of that kind run back to back (all verifies of the step, then all its
    commits, as an engine issues a step's verifies), with an event pair
    around each kind's run of launches only."""
    import torch
    import torch.distributed as dist

    by_kind = {m: [call for mm, call in calls if mm == m] for m in kinds}
    ev = {m: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)] for m in kinds}
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(steps):
        for m in kinds:
            a, b = ev[m][i]
            a.record(stream)
            for call in by_kind[m]:
                call()
            b.record(stream)
    torch.cuda.synchronize()
    return {m: statistics.fmean(a.elapsed_time(b) for a, b in ev[m]) / len(by_kind[m])
            for m in kinds}


# Single-layer workloads run as independent instances (each with its own pool
# and inputs) cycled through, all verifies before all commits: one instance's
# checkpoints fit in the 129 MB L2 on b8 (8 MiB) and b32 (64 MiB), and a commit
# issued right after its own verify would re-read them there.  In an engine the
# other layers' work runs between a layer's verify and its commit.
INSTANCES = {"b8_h16_d128_t8": 24, "b32_h32_d128_t16": 8, "b128_h32_d128_ragged16": 2}


def instances_of(name: str, requested: int = 0) -> int:
    """How many instances a run of the named workload cycles through: 1 for the
    multi-layer workload (its layers already have their own pools)."""
    if "layers" in inputs.WORKLOADS[name]:
        if requested > 1:
            raise SystemExit(f"{name} has layers of its own; --instances applies to "
                             "single-layer workloads")
        return 1
    return requested if requested > 0 else INSTANCES.get(name, 1)


def instance_note(name: str, n: int, fused: bool) -> str:
    if n == 1:
        return "1 instance"
    return (f"{n} instances (own pools and tokens), "
            + ("fused calls in turn" if fused else
               "all verifies, then all commits, so that no commit re-reads in L2 a "
               "checkpoint its verify just read"))


# The other target workloads, timed in the same run as the headline.
PER_CONFIG = [("b32_h32_d128_t16", "engine"), ("b128_h32_d128_ragged16", "fused")]


def run_per_config(args, dev, stream, world):
    """The b32 (verify+commit) and b128 ragged (fused) workloads, each timed like
    the headline: one event pair around back-to-back steps, and bracketed launches
    for the dominant kernel's roofline fraction."""
    import torch

    from speculative_decode_gated_gb300 import binding, staging

    peak, peak_kind = measured_peaks()
    out = {}
    for name, order in PER_CONFIG:
        n_inst = instances_of(name)
        why = instance_note(name, n_inst, order == "fused")
        probs = [inputs.make_problem(name, layer=l) for l in range(n_inst)]
        p0 = probs[0]
        pool = staging.new_pool(p0.pool_slots, p0.heads, p0.dk, p0.dv, dev, fill="zero",
                                layers=n_inst)
        dps = [staging.DeviceProblem(pr, dev, pool=pool[l], algo=args.algo)
               for l, pr in enumerate(probs)]
        if order == "fused":
            kinds = ["f"]
            calls = [("f", d.launcher("fused", stream)) for d in dps]
        else:
            kinds = ["v", "c"]
            calls = ([("v", d.launcher("verify", stream)) for d in dps]
                     + [("c", d.launcher("commit", stream)) for d in dps])
        bytes_of = {m: [alg_bytes(pr, MODE_NAME[m]) for pr in probs] for m in kinds}
        ms_total, avg_ms, n_per_step, ms_direct = time_calls(
            calls, kinds, stream, args.per_config_steps, args.warmup, world, dev, check=dps,
            graph=not args.no_graph)
        us_call = job_us_per_layer_call(ms_total, args.per_config_steps, n_inst, world)
        us_direct = (None if ms_direct is None else
                     job_us_per_layer_call(ms_direct, args.per_config_steps, n_inst, world))
        bytes_call = sum(sum(bytes_of[m]) for m in kinds) / n_inst
        gbs = bytes_call / (us_call * 1e-6) / 1e9
        dominant = max(kinds, key=lambda m: avg_ms[m] * n_per_step[m])
        per_launch = sum(bytes_of[dominant]) / len(bytes_of[dominant])
        achieved = per_launch / (avg_ms[dominant] * 1e-3) / 1e9
        out[name] = {
            "order": why,
            "us_per_layer_call": us_call,
            "us_per_layer_call_launched_one_by_one": us_direct,
            "alg_bytes_per_layer_call": bytes_call,
            "achieved_gbs": gbs,
            "frac_of_measured_hbm": gbs / (peak * world),
            "frac_of_8tbs": gbs / (NOMINAL_HBM_GBS * world),
            "meets_70pct_of_8tbs": gbs >= 0.7 * NOMINAL_HBM_GBS * world,
            "kernel_us": {MODE_NAME[m]: avg_ms[m] * 1e3 for m in kinds},
            "dominant": {"kernel": MODE_NAME[dominant], "achieved_gbs": achieved,
                         "frac": achieved / peak, "peak_source": peak_kind},
            "steps": args.per_config_steps,
        }
        del calls, dps, pool
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from speculative_decode_gated_gb300 import binding, staging

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.lib()  # fails loudly if the CUDA library is missing
    name = args.workload
    multi = "layers" in inputs.WORKLOADS[name]
    # layers of the multi-layer workload, or independent instances of a single-layer one
    n_layers = inputs.WORKLOADS[name]["layers"] if multi else args.instances
    if args.layers:
        n_layers = min(n_layers, args.layers)
    layers = [inputs.make_problem(name, layer=l, draft=args.draft,
                                  gate="log" if args.log_gate else "alpha", batch=args.batch)
              for l in range(n_layers)]
    L = len(layers)
    p0 = layers[0]
    pool = staging.new_pool(p0.pool_slots, p0.heads, p0.dk, p0.dv, dev, fill="zero",
                            layers=L if L > 1 else None)
    dps = [staging.DeviceProblem(pr, dev, pool=(pool[l] if L > 1 else pool), algo=args.algo,
                                 o_bf16=args.o_bf16)
           for l, pr in enumerate(layers)]
    if multi:
        staging.share_request_arrays(dps)  # one step's requests, as an engine holds them
    fused = args.mode == "fused"
    batched = args.batch_layers
    if batched and not (multi and (fused or args.order == "engine")):
        raise SystemExit("--batch-layers needs a multi-layer workload and --mode fused or "
                         "--order engine")
    if not args.no_graph:  # capture needs a stream other than the default one
        torch.cuda.set_stream(torch.cuda.Stream(dev))
    stream = torch.cuda.current_stream(dev)
    o_bytes = 2 if args.o_bf16 else 4
    per_layer = {m: [alg_bytes(pr, MODE_NAME[m], o_bytes) for pr in layers]
                 for m in ("v", "c", "f", "cv")}
    # bytes_of[kind]: algorithmic bytes of each launch of that kind in one step
    bytes_of = dict(per_layer, C=[sum(per_layer["c"])], F=[sum(per_layer["f"])])
    replay_bufs = None
    if args.replay:
        if fused or batched or args.order != "interleaved":
            raise SystemExit("--replay times verify then commit per layer")
        replay_bufs = [inputs.make_replay(pr, args.replay, seed=l, dense=False)
                       for l, pr in enumerate(layers)]
        reps = [staging.DeviceReplay(b, pr.qkv_dtype, dev) for b, pr in zip(replay_bufs, layers)]
        bytes_of["rv"] = [replay_bytes(pr, b, "verify") for pr, b in zip(layers, replay_bufs)]
        bytes_of["rc"] = [replay_bytes(pr, b, "commit") for pr, b in zip(layers, replay_bufs)]
        kinds = ["rv", "rc"]
        calls = []
        for d, r in zip(dps, reps):
            calls.append(("rv", staging.replay_launcher(d, r, "verify", stream)))
            calls.append(("rc", staging.replay_launcher(d, r, "commit", stream)))
    elif args.order == "lagged":
        if fused or batched:
            raise SystemExit("--order lagged is one call per layer and step")
        # Each layer's previous step is its own problem one step earlier (same
        # requests, tokens and accepted lengths); the W cache alternates between
        # two buffers, read by one step and written by the next.
        kinds = ["cv"]
        calls = []
        for d in dps:
            ws = [torch.zeros((d.host.n_tok, d.host.heads, d.host.dv), device=dev) for _ in range(2)]
            prevs = [binding.make_prev_step(k=d.k, alpha=d.alpha, w=ws[j], accepted=d.accepted,
                                            max_T=d.host.max_T, cu_seqlens=d.cu_seqlens)
                     for j in range(2)]
            calls.append(("cv", staging.commit_verify_launcher(d, prevs, ws, stream)))
    elif batched and fused:
        kinds = ["F"]
        calls = [("F", staging.layers_launcher(dps, "fused", stream))]
    elif batched:
        kinds = ["v", "C"]
        calls = ([("v", d.launcher("verify", stream)) for d in dps]
                 + [("C", staging.layers_launcher(dps, "commit", stream))])
    else:
        kinds = ["f"] if fused else ["v", "c"]
        if args.order == "engine" and not fused:
            order = [(d, "v") for d in dps] + [(d, "c") for d in dps]
        else:
            order = [(d, m) for d in dps for m in kinds]
        calls = [(m, d.launcher(MODE_NAME[m], stream)) for d, m in order]
    if args.with_accept:
        # The step starts with the greedy accepted lengths computed on the device
        # from token ids (one call for all layers), as an engine would.
        draft, target = inputs.make_token_ids(p0, seed=5)
        ids = [torch.from_numpy(x).to(dev) for x in (draft, target)]
        d0 = dps[0]

        def accept_call():
            binding.gdn_accept_prefix(ids[0], ids[1], d0.accepted, p0.max_T,
                                      cu_seqlens=d0.cu_seqlens, dev_err=d0.dev_err, stream=stream)
        kinds = ["a"] + kinds
        calls = [("a", accept_call)] + calls
        bytes_of["a"] = [2 * 4 * p0.n_tok + 4 * p0.batch + (4 * (p0.batch + 1) if p0.ragged else 0)]
    bytes_call = sum(sum(bytes_of[m]) for m in kinds) / L

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ms_total, avg_ms, n_per_step, ms_direct = time_calls(
        calls, kinds, stream, args.steps, args.warmup, world, dev, check=dps,
        graph=not args.no_graph)
    b2b = None
    if len(kinds) > 1 and not args.replay:
        b2b = time_back_to_back(calls, kinds, stream, args.steps, world, dev)
    clk = clocks.stop()
    ms_step = ms_total / args.steps
    us_call = job_us_per_layer_call(ms_total, args.steps, L, world)
    us_direct = None if ms_direct is None else job_us_per_layer_call(ms_direct, args.steps, L, world)

    dominant = max(kinds, key=lambda m: avg_ms[m] * n_per_step[m])
    per_launch_bytes = {m: sum(bytes_of[m]) / len(bytes_of[m]) for m in kinds}
    peak, peak_kind = measured_peaks()
    achieved = per_launch_bytes[dominant] / (avg_ms[dominant] * 1e-3) / 1e9
    algo_used = binding.gdn_select_algo(dps[0].c)
    ktag = ({binding.GDN_ALGO_CHUNK: "gdn_chunk", binding.GDN_ALGO_CHUNK_TC: "gdn_chunk_tc"}
            .get(algo_used, "gdn_recurrent") + "_" + MODE_NAME[dominant])
    # the committed captures are of the named workloads' own launches (default
    # instantiation, full layer count); a changed shape or variant has none
    traffic = (None if (args.batch or args.draft or args.o_bf16 or args.log_gate or args.replay
                        or (batched and args.layers))
               else profile_traffic(ktag, name))

    e2e = (run_e2e(args, dps, stream, dev, fused, world)
           if not (args.no_e2e or batched or args.replay or args.order == "lagged") else None)
    per_config = None
    if not (args.no_per_config or args.replay or args.draft or args.batch or args.layers or batched
            or args.order != "interleaved" or args.workload != WORKLOAD
            or args.o_bf16 or args.log_gate):
        per_config = run_per_config(args, dev, stream, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.replay:
        threads = os.cpu_count() or 1
        dt, us, n = cpu_oracle_time(p0, args.cpu_units, threads)
        cpu = {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} of {p0.units} units of layer 0, verify pass + commit pass, "
                         f"{dt:.1f} s wall, scaled to a full layer-call"}
        if args.cpu_units_1t > 0:
            dt1, us1, n1 = cpu_oracle_time(p0, args.cpu_units_1t, 1)
            cpu["single_thread"] = {
                "value": us1, "unit": UNIT, "cores": 1,
                "sample": f"{n1} of {p0.units} units of layer 0, {dt1:.1f} s wall, "
                          f"scaled to a full layer-call"}

    if rank == 0:
        gbs = bytes_call / (us_call * 1e-6) / 1e9  # the whole job's GB/s
        line = {
            "metric": METRIC, "value": us_call, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {
                "workload": name if args.batch is None else f"{name} with batch {p0.batch}",
                "description": (f"batch {p0.batch}, heads {p0.heads}, dk {p0.dk}, dv {p0.dv}, "
                                f"draft {p0.max_T}, "
                                + (f"{L} layer(s)" if multi else
                                   instance_note(name, L, fused and not args.replay))
                                + f", pool {p0.pool_slots} slots/layer, "
                                f"q/k/v {p0.qkv_dtype}, gates/state/o fp32"),
                "order": (f"ReplaySSM buffer of {args.replay} rows per slot: replay verify then "
                          "replay commit per layer; buffered lengths uniform on [0, C - T] "
                          "(a steady-state sample, not carried between steps)" if args.replay else
                          "fused, all layers in one launch" if fused and batched else
                          "fused per layer" if fused else
                          "all verifies, then all layers' commits in one launch" if batched else
                          "verify then commit per layer" if args.order == "interleaved" else
                          "per layer: commit the previous step, verify this one (one call)"
                          if args.order == "lagged" else
                          "all verifies then all commits"),
                "l2": "inputs larger than L2 (each step touches ~%.1f GB)" % (bytes_call * L / 1e9),
                "issue": ("each timed step replays the step's calls captured once in a CUDA graph "
                          "(value_launched_one_by_one: the same calls launched one by one)"
                          if us_direct is not None else "the calls launched one by one"),
                "algo": {1: "recurrent", 2: "chunk", 3: "chunk_tc"}.get(algo_used, str(algo_used)),
                "arith": ("fp32 state and outputs; the state-sized products on tensor cores "
                          "in bf16 on hi/lo splits of the fp32 operands (about 16 mantissa "
                          "bits), fp32 accumulation; solves and gates in fp32"
                          if algo_used in (binding.GDN_ALGO_CHUNK, binding.GDN_ALGO_CHUNK_TC)
                          else "fp32 on CUDA cores"),
                "accepted": ("greedy prefix match of token ids on the device, every step"
                             if args.with_accept else "given (device array)"),
                "variant": ", ".join(v for v, on in (("bf16 o", args.o_bf16),
                                                     ("log-space gates", args.log_gate)) if on)
                           or "none",
            },
            "value_launched_one_by_one": us_direct,
            "achieved_gbs": gbs,
            "frac_of_8tbs": gbs / (NOMINAL_HBM_GBS * world),
            "frac_of_measured_hbm": gbs / (peak * world),
            "alg_bytes_per_layer_call": bytes_call,
            "kernel_us": {MODE_NAME[m]: avg_ms[m] * 1e3 for m in kinds},
            "kernel_us_back_to_back": None if b2b is None else dict(
                {MODE_NAME[m]: b2b[m] * 1e3 for m in kinds},
                how="mean per launch when the step's launches of one kind run back to back "
                    "(events around each kind's run only); kernel_us brackets every launch "
                    "with events, which breaks the dependent-launch overlap"),
            "roofline": {"bound": "hbm", "kernel": ktag, "achieved": achieved, "peak": peak,
                         "peak_source": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "alg_bytes_per_launch": per_launch_bytes[dominant]},
            "gpu_launches": args.steps * len(calls),  # in timed region 1
            "clocks": clk,
            "e2e": e2e,
            "per_config": per_config,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_e2e(args, dps, stream, dev, fused, world=1):
    """Same metric end to end: every step copies each layer's q/k/v/gates/accepted
    from pinned host memory and reads every layer's o back, overlapped on copy
    streams with the kernels of other layers.  With N ranks, the slowest rank's
    time over all ranks' layer-calls, and the copied bytes of all ranks."""
    import torch

    # Each layer's inputs live in one device buffer (q, k, v, alpha, beta and the
    # accepted lengths as 16-byte-aligned views of it) filled from one pinned host
    # buffer: one host-to-device copy per layer and step.
    names = ("q", "k", "v", "alpha", "beta", "accepted")
    host_in, dev_in = [], []
    for d in dps:
        parts = [getattr(d, n) for n in names]
        nbytes = [t.numel() * t.element_size() for t in parts]
        offs, total = [], 0
        for nb in nbytes:
            offs.append(total)
            total += (nb + 15) // 16 * 16
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        for n, t, off, nb in zip(names, parts, offs, nbytes):
            view = dbuf[off:off + nb].view(t.dtype).view(t.shape)
            view.copy_(t)
            hbuf[off:off + nb].copy_(t.cpu().contiguous().view(torch.uint8).view(-1))
            setattr(d, n, view)
        d.c = d._make_c()  # the C problem now points into the packed buffer
        host_in.append(hbuf)
        dev_in.append(dbuf)
    host_o = [torch.empty(d.o.shape, dtype=d.o.dtype).pin_memory() for d in dps]
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    L = len(dps)
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_used = [torch.cuda.Event() for _ in range(L)]
    ev_o = [torch.cuda.Event() for _ in range(L)]
    ev_read = [torch.cuda.Event() for _ in range(L)]
    bi = sum(h.numel() for h in host_in)
    bo = sum(t.numel() * t.element_size() for t in host_o)
    kinds = ["fused"] if fused else ["verify", "commit"]
    calls = [{m: d.launcher(m, stream) for m in kinds} for d in dps]

    def one_step():
        for l, d in enumerate(dps):
            with torch.cuda.stream(h2d):
                h2d.wait_event(ev_used[l])
                dev_in[l].copy_(host_in[l], non_blocking=True)
                ev_in[l].record(h2d)
            stream.wait_event(ev_in[l])
            stream.wait_event(ev_read[l])
            if fused:
                calls[l]["fused"]()
                ev_o[l].record(stream)
            else:
                calls[l]["verify"]()
                ev_o[l].record(stream)
                calls[l]["commit"]()
            ev_used[l].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_o[l])
                host_o[l].copy_(d.o, non_blocking=True)
                ev_read[l].record(d2h)

    for _ in range(max(args.warmup, 1)):
        one_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one_step()
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, world, dev)

    # The host link's floor for the same bytes: the same copies, both directions
    # at once on the two copy streams, with no kernel running.
    def copies_only():
        for l, d in enumerate(dps):
            with torch.cuda.stream(h2d):
                dev_in[l].copy_(host_in[l], non_blocking=True)
            with torch.cuda.stream(d2h):
                host_o[l].copy_(d.o, non_blocking=True)

    copies_only()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        copies_only()
    torch.cuda.synchronize()
    dt_copy = max_over_ranks(time.perf_counter() - t0, world, dev)
    floor = job_us_per_layer_call(dt_copy * 1e3, args.e2e_steps, L, world)
    return {"value": job_us_per_layer_call(dt * 1e3, args.e2e_steps, L, world), "unit": UNIT,
            "h2d_bytes_per_step": bi * world, "d2h_bytes_per_step": bo * world,
            "steps": args.e2e_steps,
            "copy_floor": {"value": floor, "unit": UNIT,
                           "link_gbs": (bi + bo) / (dt_copy / args.e2e_steps) / 1e9,
                           "how": "the same host<->device copies alone, both directions at "
                                  "once, no kernels: the host link bounds the end-to-end "
                                  "figure from below"}}


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--mode", choices=["separate", "fused"], default=None,
                    help="separate verify + commit (default) or the fused call")
    ap.add_argument("--order", choices=["interleaved", "engine", "lagged"], default=None,
                    help="separate calls: verify then commit per layer (interleaved; the "
                         "default for the multi-layer workload), all verifies then all commits "
                         "(engine; the default for instances of a single-layer workload), or "
                         "one commit-then-verify call per layer (lagged)")
    ap.add_argument("--instances", type=int, default=0,
                    help="independent instances of a single-layer workload cycled through "
                         "(0: the workload's default, enough that no commit finds its "
                         "checkpoints in L2)")
    ap.add_argument("--algo", type=int, default=0,
                    help="0 auto, 1 recurrent, 2 chunk (mma.sync), 3 chunk (tcgen05)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (small cases for profiling; 0 = all)")
    ap.add_argument("--cpu-units", type=int, default=256)
    ap.add_argument("--cpu-units-1t", type=int, default=32,
                    help="units of the single-threaded oracle sample (0 skips it)")
    ap.add_argument("--ref-units", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--replay", type=int, default=0, metavar="C",
                    help="time the ReplaySSM buffer calls with C buffer rows per slot")
    ap.add_argument("--batch", type=int, default=None,
                    help="replace the number of requests of a uniform workload (a sweep of "
                         "the unit count against the 304 resident blocks)")
    ap.add_argument("--draft", type=int, default=None,
                    help="replace the draft length of a uniform workload (longer drafts run as "
                         "several 16-token chunks)")
    ap.add_argument("--with-accept", action="store_true",
                    help="start every step with the on-device greedy accept-length call")
    ap.add_argument("--batch-layers", action="store_true",
                    help="all layers' commits (or fused calls) in one layer-batch launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--o-bf16", action="store_true", help="the bf16-output variant")
    ap.add_argument("--log-gate", action="store_true", help="the log-space gate variant")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the headline loop with the calls launched one by one (default: "
                         "replays of one step captured in a CUDA graph; the one-by-one figure "
                         "is reported beside it)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the b32 and b128 ragged workloads timed after the headline")
    ap.add_argument("--per-config-steps", type=int, default=200)
    args = ap.parse_args()
    if args.mode is None:
        args.mode = "fused" if "ragged" in args.workload else "separate"
    args.instances = instances_of(args.workload, args.instances)
    if args.order is None:
        args.order = "engine" if args.instances > 1 and not args.replay else "interleaved"
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
