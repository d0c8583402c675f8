#!/usr/bin/env python
"""Benchmark of the GB300 decode projection y[B,N] = BF16(x[B,K] . W[N,K]^T).

One step = one pass of the projection over every call of the workload (default:
the o_proj sweep, x[B,12288] . W[7168,12288]^T for B = 1, 2, 4, 8, 16 with seeds
0..4, i.e. five distinct 176 MB weights).  Inputs are resident in HBM before the
timed region; every weight is larger than the 129 MB L2 and each step cycles
five of them, so no weight is served from L2.  The metric is achieved HBM
bandwidth: algorithmic bytes (W + x + y of every call) per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     # the CPU oracle on a bounded sample

Prints one JSON line (rank 0).  Under torchrun each rank runs the same
workload on its own GPU (replicas: the projection has no exchange step) and
the line reports the total bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from skinny_bf16_split_gb300 import synth  # noqa: E402

METRIC = "achieved HBM GB/s (% of peak) and µs/call, BF16 decode projection B=1–256"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_TEXT = {
    "oproj_sweep": "o_proj sweep: x[B,12288] . W[7168,12288]^T, B in {1,2,4,8,16}, seeds 0..4",
    "dsa_b1": "DSA packed input projection: x[1,7168] (unit-RMS rows) . W[14560,7168]^T, seed 0",
    "kda_sweep": "KDA packed input projection: x[B,7168] . W[49376,7168]^T, B in {1,4,8,16}, seeds 0..3",
    "dsa_wide": "wide DSA input projection: x[B,7168] . W[14560,7168]^T, B in {32,64,128,256}, seeds 0..3",
    "chain": "8-layer decode chain: per layer x[16,7168] . W_dsa[14560,7168]^T then "
             "x'[16,12288] . W_o[7168,12288]^T, 16 distinct weights, seed 7",
    "dsa_verify": "verify-step batches on the DSA input projection: x[B,7168] . W[14560,7168]^T, "
                  "B = requests x q in {3,6,12,24,48}, seeds 0..4, tuned plan",
    "tp_sharded": "TP-G shards at B=16: DSA input projection rows 14560/G x 7168 and o_proj "
                  "7168 x 12288/G for G in {2,4,8}, seeds 0..5, tuned plan",
}
# Workloads whose plan is tuned by default (the verify-step tables are measured).
TUNED_BY_DEFAULT = {"dsa_verify", "tp_sharded"}
# Sources each kernel family is built from (a traffic record is stale once they change).
KERNEL_SOURCES = {"splitk_fma": ["splitk_fma.cu"], "tc_gemm": ["tc_gemm.cu", "exchange.cuh"],
                  "tc_split": ["tc_split.cu", "exchange.cuh"], "rows_gemv": ["rows_gemv.cu"],
                  "tc_wide": ["tc_wide.cu"], "tc_cluster": ["tc_cluster.cu"]}
SHARED_SOURCES = ["ptx.cuh", "internal.h"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=synth.WORKLOADS, default="oproj_sweep")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="wall-clock budget of the oracle CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--plan", default="default", choices=("default", "tune"))
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay (programmatic dependent launch) measurement")
    ap.add_argument("--report", action="store_true",
                    help="measure every workload; one JSON line each (per-config report)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float) -> float:
    """The largest `value` over all ranks (the value itself when not distributed).
    Works on the NCCL (CUDA tensor) and gloo (CPU tensor) backends."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    device = "cuda" if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Throughput of the whole job: the bytes every rank moved over the slowest
    rank's time (each rank runs the same workload: weak scaling)."""
    return bytes_per_step * steps * world / (elapsed_ms * 1e-3) / 1e9


def source_hash(family: str | None = None) -> str:
    """Hash of a kernel family's sources (all families when None)."""
    names = ([n for v in KERNEL_SOURCES.values() for n in v] if family is None
             else KERNEL_SOURCES[family]) + SHARED_SOURCES
    h = hashlib.sha256()
    for name in names:
        p = os.path.join(ROOT, "skinny_bf16_split_gb300", "csrc", name)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def kernel_family(kernel: str) -> str:
    return next(f for f in KERNEL_SOURCES if kernel.startswith(f))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    try:
        fields = dict(line.split(":", 1) for line in open(path) if ":" in line)
    except OSError:
        return None
    if fields.get("source_sha", "").strip() != source_hash(kernel_family(kernel)):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks -----

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.device = device_index

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            target = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", target, f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1].split()[0]), float(parts[2].split()[0]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------- cpu baseline ----

def cpu_baseline(calls, weights, xs, seconds: float):
    """The oracle timed on this host's cores over a bounded sample of rows of
    every call; returns bytes/s in GB/s over the sample."""
    import oracle
    threads = oracle.max_threads()
    oracle.linear_rows(xs[0], weights[calls[0].weight_key], np.arange(4), threads)  # warm
    per_call = seconds / len(calls)
    done_bytes, done_time, rows_total = 0, 0.0, 0
    for c, x in zip(calls, xs):
        W = weights[c.weight_key]
        rows, t_call, start = 32, 0.0, 0
        while t_call < per_call and start < c.N:
            idx = np.arange(start, min(c.N, start + rows))
            t0 = time.perf_counter()
            oracle.linear_rows(x, W, idx, threads)
            dt = time.perf_counter() - t0
            t_call += dt
            done_bytes += 2 * (idx.size * c.K + c.B * c.K + c.B * idx.size)
            rows_total += idx.size
            start += idx.size
            rows = max(32, min(4 * rows, int(rows * (per_call - t_call) / max(dt, 1e-6))))
        done_time += t_call
    return {"value": done_bytes / done_time / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows_total} weight rows in total across the {len(calls)} calls "
                      f"(all B rows of x each), ~{seconds:.0f} s of oracle work, exact integer "
                      f"accumulation, OpenMP over outputs"}


# ------------------------------------------------------------ reference arm ---

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    calls = synth.workload(args.workload)
    threads = oracle.max_threads()
    weights, xs = {}, []
    for c in calls:
        if c.weight_key not in weights:
            weights[c.weight_key] = c.weight()
        xs.append(c.activations())
    # calibrate rows per call so the whole run stays within about a minute
    per_row = []
    for c, x in zip(calls, xs):
        t0 = time.perf_counter()
        oracle.linear_rows(x, weights[c.weight_key], np.arange(min(c.N, 64)), threads)
        per_row.append((time.perf_counter() - t0) / min(c.N, 64))
    step_budget = min(2.0, 60.0 / max(1, args.steps + args.warmup))
    rows = [max(1, min(c.N, int(step_budget / len(calls) / max(p, 1e-9)))) for c, p in zip(calls, per_row)]
    idx = [np.arange(r) for r in rows]
    step_bytes = sum(2 * (r * c.K + c.B * c.K + c.B * r) for c, r in zip(calls, rows))

    def step():
        for c, x, i in zip(calls, xs, idx):
            oracle.linear_rows(x, weights[c.weight_key], i, threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    elapsed = time.perf_counter() - t0
    value = step_bytes * args.steps / elapsed / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(args.workload, calls),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step the first {rows} weight rows of each call "
                                   f"(all B rows of x)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(name, calls):
    return {"workload": WORKLOAD_TEXT[name],
            "shapes": sorted({f"N={c.N},K={c.K}" for c in calls}),
            "batches": [c.B for c in calls], "accumulate": "fp32", "output": "bf16",
            "l2": "inputs larger than L2: every call streams its own >=176 MB weight (L2 is 129 MB)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- our arm ----

def kernel_name(t) -> str:
    import skinny_bf16_split_gb300 as dep
    if t.kind == dep.DEP_KIND_SPLITK_FMA:
        return f"splitk_fma_c{t.cols}"
    if t.kind == dep.DEP_KIND_ROWS:
        return f"rows_gemv_c{t.cols}"
    if t.kind == dep.DEP_KIND_TC_SPLIT:
        return f"tc_split_n{t.cols}"
    if t.kind == dep.DEP_KIND_TC_WIDE:
        return f"tc_wide_n{t.cols}_g{t.tile_n // 128}"
    if t.kind == dep.DEP_KIND_TC_CLUSTER:
        return f"tc_cluster_n{t.cols}_g{t.tile_n // 128}_k{t.splits}"
    return f"tc_gemm_n{t.cols}"


def run_ours(args):
    import torch
    import skinny_bf16_split_gb300 as dep

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.cuda.current_device()
    dep.lib()  # fails loudly when the library is not built

    calls = synth.workload(args.workload)
    weights, xs_host = {}, []
    for c in calls:
        if c.weight_key not in weights:
            weights[c.weight_key] = c.weight()
        xs_host.append(c.activations())

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)

    W_dev = {k: dev(v) for k, v in weights.items()}
    x_dev = [dev(x) for x in xs_host]
    y_dev = [torch.empty((c.B, c.N), dtype=torch.bfloat16, device=device) for c in calls]
    plans = {}
    for c in calls:
        plans.setdefault((c.N, c.K), set()).add(c.B)
    tuned = args.plan == "tune" or args.workload in TUNED_BY_DEFAULT
    flags = dep.DEP_PLAN_TUNE if tuned else dep.DEP_PLAN_DEFAULT
    plans = {k: dep.dep_projection_plan(k[0], k[1], sorted(v), flags) for k, v in plans.items()}
    tactics = [dep.dep_projection_plan_query(plans[(c.N, c.K)], c.B) for c in calls]
    launches_per_step = sum(-(-c.B // t.cols) for c, t in zip(calls, tactics))
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    bytes_per_step = sum(c.algorithmic_bytes for c in calls)
    lib = dep.lib()
    args_c = [(plans[(c.N, c.K)], x_dev[i].data_ptr(), W_dev[c.weight_key].data_ptr(),
               y_dev[i].data_ptr(), c.B) for i, c in enumerate(calls)]

    def one_step(ev=None):
        for i, (p, x, W, y, B) in enumerate(args_c):
            if ev is not None:
                ev[i][0].record(stream)
            st = lib.dep_projection_run(p, x, W, y, B, sptr)
            if st:
                raise dep.DepError(st, "dep_projection_run")
            if ev is not None:
                ev[i][1].record(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(device)
    sampler.start()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(args.warmup):
        one_step()
    w1.record(stream)
    torch.cuda.synchronize()
    step_ms_est = w0.elapsed_time(w1) / max(1, args.warmup)
    lead = run_ahead_steps(step_ms_est, launches_per_step + 1)              # value region
    lead_ev = run_ahead_steps(step_ms_est, launches_per_step + 2 * len(calls))  # per-call events

    # Timed region for `value`: K steps back to back, CUDA events at its two ends
    # only (a pair of events around every call costs the GPU front end a few us
    # per call, which a decode step does not pay).  Host run-ahead is bounded
    # with one untimed marker event per step.
    marks = [torch.cuda.Event() for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(args.steps):
        one_step()
        marks[s].record(stream)
        if s >= lead:  # keep the host a bounded number of steps ahead of the GPU
            marks[s - lead].synchronize()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = t_start.elapsed_time(t_end)

    # Instrumented region: the same K steps with every call bracketed by its own
    # events, for the per-call figures and the dominant kernel's launch duration.
    events = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in calls] for _ in range(args.steps)]
    i_start, i_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    i_start.record(stream)
    for s in range(args.steps):
        one_step(events[s])
        if s >= lead_ev:
            events[s - lead_ev][-1][1].synchronize()
    i_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    instrumented_ms = reduce_max(i_start.elapsed_time(i_end))
    call_ms = np.array([[events[s][i][0].elapsed_time(events[s][i][1]) for i in range(len(calls))]
                        for s in range(args.steps)])
    for p in plans.values():
        code = dep.dep_projection_device_status(p)
        if code:
            raise RuntimeError(f"a kernel reported device status {code}")
    elapsed_ms = reduce_max(elapsed_ms)
    value = whole_job_gbs(bytes_per_step, args.steps, world, elapsed_ms)
    peak, peak_src = read_peaks()

    # per-kernel totals over the timed region; the dominant kernel's roofline
    per_kernel = {}
    for i, (c, t) in enumerate(zip(calls, tactics)):
        k = kernel_name(t)
        d = per_kernel.setdefault(k, {"ms": 0.0, "bytes": 0, "launches": 0})
        d["ms"] += float(call_ms[:, i].sum())
        d["bytes"] += c.algorithmic_bytes * args.steps
        d["launches"] += -(-c.B // t.cols) * args.steps
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    d = per_kernel[dom]
    achieved_bracketed = d["bytes"] / (d["ms"] * 1e-3) / 1e9

    # The dominant kernel's launch duration: its calls alone, K steps back to
    # back on the launching stream, CUDA events at the two ends of the region.
    dom_calls = [i for i, t in enumerate(tactics) if kernel_name(t) == dom]
    d_start, d_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    d_start.record(stream)
    for s in range(args.steps):
        for i in dom_calls:
            p, x, W, y, B = args_c[i]
            st = lib.dep_projection_run(p, x, W, y, B, sptr)
            if st:
                raise dep.DepError(st, "dep_projection_run")
        marks[s].record(stream)
        if s >= lead:
            marks[s - lead].synchronize()
    d_end.record(stream)
    torch.cuda.synchronize()
    dom_ms = reduce_max(d_start.elapsed_time(d_end))
    achieved = d["bytes"] / (dom_ms * 1e-3) / 1e9
    traffic = read_traffic(dom, args.workload)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "peak_source": f"{peak_src} (HBM copy bandwidth)",
                "bytes_per_launch": d["bytes"] / d["launches"],
                "us_per_launch": dom_ms * 1e3 / d["launches"],
                "duration_timing": "the kernel's calls alone, K steps back to back, CUDA events at the "
                                   "region's ends",
                "achieved_with_per_call_events": achieved_bracketed,
                "share_of_timed_region": d["ms"] / (call_ms.sum() or 1.0)}
    per_call = []
    for i, (c, t) in enumerate(zip(calls, tactics)):
        # Event timestamps tick in about 2 us steps: the mean over the timed
        # steps resolves a call's time, a single pair (or the median) does not.
        us = float(np.mean(call_ms[:, i])) * 1e3
        per_call.append({"call": c.name, "N": c.N, "K": c.K, "B": c.B, "us_mean": us,
                         "us_median": float(np.median(call_ms[:, i])) * 1e3,
                         "gbs": c.algorithmic_bytes / (us * 1e-6) / 1e9,
                         "frac_of_peak": c.algorithmic_bytes / (us * 1e-6) / 1e9 / peak,
                         "kernel": kernel_name(t), "tactic": t.as_dict()})

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, dep, calls, plans, xs_host, W_dev, device, world)
    graph = None
    if not args.no_graph:
        graph = run_graph_pdl(args, dep, calls, x_dev, W_dev, y_dev, device, world, flags)

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(calls, weights, xs_host, args.cpu_seconds)

    for p in plans.values():
        dep.dep_projection_plan_destroy(p)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload, calls),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "graph_pdl": graph,
            "timing": "value: K steps back to back, CUDA events at the region's ends only; per_call: "
                      "the same K steps again with every call bracketed by its own events "
                      f"({instrumented_ms / args.steps:.4f} ms per step with those events)",
            "gpu_launches": launches_per_step * args.steps, "per_call": per_call,
            "plan": "tune" if tuned else "default", "kernel_sources": source_hash(),
            "device": torch.cuda.get_device_name(device),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_ahead_steps(step_ms: float, entries_per_step: int) -> int:
    """Steps the host may enqueue ahead of the GPU in a timed loop: about 20 ms
    of queued work, and at most about 400 queued operations.  Enough that a
    host thread descheduled for a few ms does not let the GPU run dry, few
    enough that the launch queue never fills (a full queue blocks the host
    inside a launch call, and a host woken late from that block lets the GPU
    drain in the middle of a timed call)."""
    by_time = int(np.ceil(20.0 / max(step_ms, 1e-3)))
    by_queue = 400 // max(1, entries_per_step)
    return max(2, min(by_time, by_queue))


def run_graph_pdl(args, dep, calls, x_dev, W_dev, y_dev, device, world, flags):
    """One step captured as a CUDA graph on plans with programmatic dependent
    launch (each kernel streams its first weight tiles while the previous one
    finishes), replayed K times; events around all replays."""
    import torch
    keys = {}
    for c in calls:
        keys.setdefault((c.N, c.K), set()).add(c.B)
    plans = {k: dep.dep_projection_plan(k[0], k[1], sorted(v), flags | dep.DEP_PLAN_PDL)
             for k, v in keys.items()}
    lib = dep.lib()
    stream = torch.cuda.Stream()
    run_args = [(plans[(c.N, c.K)], x_dev[i].data_ptr(), W_dev[c.weight_key].data_ptr(),
                 y_dev[i].data_ptr(), c.B) for i, c in enumerate(calls)]

    def step(sptr):
        for p, x, W, y, B in run_args:
            st = lib.dep_projection_run(p, x, W, y, B, sptr)
            if st:
                raise dep.DepError(st, "dep_projection_run")

    with torch.cuda.stream(stream):
        step(stream.cuda_stream)  # eager warm-up (kernel attributes, descriptors)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(stream.cuda_stream)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    cur = torch.cuda.current_stream()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(cur)
    graph.replay()
    w1.record(cur)
    torch.cuda.synchronize()
    lead = run_ahead_steps(w0.elapsed_time(w1), 2)
    marks = [torch.cuda.Event() for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for s in range(args.steps):
        graph.replay()
        marks[s].record(cur)
        if s >= lead:
            marks[s - lead].synchronize()
    t1.record(cur)
    torch.cuda.synchronize()
    ms = reduce_max(t0.elapsed_time(t1))
    for p in plans.values():
        code = dep.dep_projection_device_status(p)
        if code:
            raise RuntimeError(f"a kernel reported device status {code}")
        dep.dep_projection_plan_destroy(p)
    bytes_per_step = sum(c.algorithmic_bytes for c in calls)
    return {"value": whole_job_gbs(bytes_per_step, args.steps, world, ms), "unit": UNIT,
            "ms_per_step": ms / args.steps,
            "how": "one step captured as a CUDA graph, kernels chained by programmatic dependent "
                   "launch (DEP_PLAN_PDL), K replays timed by events"}


def run_e2e(args, dep, calls, plans, xs_host, W_dev, device, world):
    """The same steps through dep_projection_run_host: x copied from pinned
    host memory to the device and y read back, every call of every step, and the
    step's results synchronised to the host before the next step."""
    import torch
    xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs_host]
    yh = [torch.empty((c.B, c.N), dtype=torch.bfloat16).pin_memory() for c in calls]
    stream = torch.cuda.current_stream()
    lib = dep.lib()
    args_c = [(plans[(c.N, c.K)], xh[i].data_ptr(), W_dev[c.weight_key].data_ptr(), yh[i].data_ptr(),
               c.B) for i, c in enumerate(calls)]

    def step():
        for p, x, W, y, B in args_c:
            st = lib.dep_projection_run_host(p, x, W, y, B, stream.cuda_stream)
            if st:
                raise dep.DepError(st, "dep_projection_run_host")
        stream.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    if world > 1:
        torch.distributed.barrier()
    steps = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(t_start.elapsed_time(t_end))
    bytes_per_step = sum(c.algorithmic_bytes for c in calls)
    return {"value": whole_job_gbs(bytes_per_step, steps, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": sum(2 * c.B * c.K for c in calls),
            "d2h_bytes_per_step": sum(2 * c.B * c.N for c in calls),
            "ms_per_step": ms / steps, "api": "dep_projection_run_host"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.report:
        for name in synth.WORKLOADS:
            args.workload = name
            run_ours(args)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
