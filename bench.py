#!/usr/bin/env python
"""Benchmark of the Dion3 optimizer step on GB300 (one rank per GPU).

Default workload: the 7B-shaped matrix set (d = 4096, 32 layers: 128 x
4096x4096, 64 x 4096x11008, 32 x 11008x4096; bf16 parameters and gradients,
fp32 momentum) stepped at f = 1/4, as three shape groups in one dion3_step.
A "step" is one full Dion3 optimizer step over every matrix of the set:
momentum accumulation + l1 selection, gather/normalise, fp16 Gram
Newton-Schulz (T = 5, restart at 3) and the row-scatter update.

Printed (rank 0, one JSON line):
  value        useful TFLOP/s of the whole job (Gram-NS FLOPs with a triangle
               counted as half, summed over all ranks' matrices) / max-over-
               ranks step time; inputs resident in HBM (65 GB, far above L2).
  e2e          the same metric when every step also copies its gradients from
               pinned host memory and reads the selected row indices back.
  roofline     the dominant kernel of the timed region (CUDA events around each
               memory-bound launch and each chain of GEMM launches, via the
               library's launch trace) against the measured peak in
               MEASURED_PEAKS.json.
  cpu_baseline the float64 CPU oracle timed on a bounded sample (one matrix of
               each shape group) and scaled to the full set.
  step_roofline  t_roof = useful FLOPs / sustained tensor peak + algorithmic
               bytes of the memory-bound kernels / measured copy bandwidth,
               and t_roof / measured step time (frac; frac_graph for the
               graph replay).
  graph        the same step captured once in a CUDA graph and replayed.
  paths        the two parts of the step against their own rooflines: the
               Gram-NS path (all GEMM launches) in useful TFLOP/s as a fraction
               of the measured sustained and burst bf16 peaks, and the
               select/update path (the memory-bound kernels) in GB/s as a
               fraction of the measured HBM copy bandwidth.
  per_model    (default workload only) step ms and useful TFLOP/s with their
               fraction of the measured bf16 peak for each model at each f:
               7B at f = 1/4 (the headline) and 1/8, 1B at f = 1, 1/2, 1/4,
               each with its `paths` fractions (3 extra traced steps).

--impl reference times the CPU oracle (the only reference this method has:
there is no reference implementation to install) on the same workload and
metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import select
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Dion3 optimizer-step ms & useful TFLOP/s (frac of GB300 FP16 peak) per model at f"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------

def workload_groups(name: str, max_batch: int = 0):
    """[(rows, cols, batch, param_dtype, grad_dtype)] and a description.
    ``max_batch`` > 0 caps each group's matrix count (a small case of the same
    shapes, for profiler captures)."""
    import workloads
    if name in ("7b", "1b"):
        spec = workloads.MODEL_SETS[name]
        groups = [(r, c, min(b, max_batch) if max_batch > 0 else b, "bf16", "bf16")
                  for (r, c, b) in workloads.model_groups(name)]
        desc = (f"{name.upper()}-shaped matrix set (d={spec['d']}, {spec['layers']} layers: "
                + ", ".join(f"{b}x {r}x{c}" for (r, c, b, _, _) in groups) + ")")
        return groups, desc
    if name == "gapped":
        return [(1024, 4096, 1, "bf16", "bf16")], "one 1024x4096 matrix (gapped l1 ladder)"
    if name == "single":
        return [(256, 1024, 1, "f32", "f32")], "one fp32 256x1024 matrix"
    raise SystemExit(f"unknown workload {name}")


def workload_config(args, groups, desc):
    """The `config` object of the JSON line: the workload only, the same for our
    arm and the reference arm."""
    nbytes = {"bf16": 2, "f32": 4}
    resident = sum(r * c * b * (nbytes[pd] + nbytes[gd] + 4) for (r, c, b, pd, gd) in groups)
    return {"workload": f"{desc}, f={args.f}", "f": args.f,
            "matrices": sum(g[2] for g in groups),
            "params_per_gpu": sum(g[0] * g[1] * g[2] for g in groups),
            "param_dtype": groups[0][3], "grad_dtype": groups[0][4], "momentum_dtype": "f32",
            "ns": f"Gram NS T=5 restart@3, {args.ns_dtype} operands",
            "momentum_decay": "lazy (dion3_step_lazy)" if args.lazy_decay else "eager (dion3_step)",
            "normuon": "per-neuron normalisation (dion3_step_normuon, NorMuon reading)" if args.normuon else None,
            "l2": (f"inputs larger than L2 ({resident / 1e9:.1f} GB of W, G, M resident in HBM against 129 MB)"
                   if resident > 129e6 else
                   f"inputs ({resident / 1e6:.1f} MB) smaller than L2 and not flushed between steps "
                   "(a small parity workload, not the default line)")}


def useful_flops_total(groups, f, hp_kwargs, d3):
    hp = d3.HParams(f=f, **hp_kwargs)
    tot = 0.0
    for (r, c, b, _, _) in groups:
        k = d3.num_selected(f, r)
        tot += b * d3.useful_flops(k, c, hp)
    return tot


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel: str, workload: dict = None):
    """DRAM traffic per launch of `kernel` from a committed ncu summary, or None
    if none exists, the kernel source changed since it was taken, or (when
    `workload` is given) the record was taken on another workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(kernel)
    if not rec:
        return None
    if workload is not None and rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, rec["source"])
    with open(src, "rb") as fh:
        if hashlib.sha256(fh.read()).hexdigest() != rec["source_sha256"]:
            return None
    return rec


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        """Starts sampling and waits (at most 5 s) for the first sample, so the
        sampler is running when the timed region begins; that first sample is
        kept apart, as a fallback for regions shorter than the sampling period."""
        self.first = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
        if ready:
            self.first = self.proc.stdout.readline()

    @staticmethod
    def _summary(lines):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in (ln.split(",") for ln in lines if ln.strip()):
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        got = self._summary(out.strip().splitlines())
        if got is None and self.first:
            got = self._summary([self.first])
            if got is not None:
                got["note"] = ("timed region shorter than the 100 ms sampling period: the sample taken "
                               "just before it")
        return got


# ---------------------------------------------------------------------------
# Multi-rank helpers (one process per GPU; the unit of work, one matrix, is
# independent, so ranks share nothing on the data path: weak scaling).
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device) -> float:
    """The largest `value` over all ranks (the job's time is its slowest
    rank's); `device` is where the reduction tensor lives (cuda for NCCL,
    cpu for gloo)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job useful TFLOP/s: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def traffic_workload(args) -> dict:
    """The key a traffic record is taken on: workload, f, operand type and
    matrices per group (0: the whole set)."""
    return {"workload": args.workload, "f": args.f, "ns_dtype": args.ns_dtype, "max_batch": args.max_batch}


def gemm_totals(trace: dict) -> dict:
    """Launches, time and useful FLOPs of every GEMM entry of a launch trace
    together (one entry per Newton-Schulz chain, or one per role with
    DION3_TRACE_DETAIL)."""
    return {k: sum(v[k] for v in trace.values() if v["useful_flops"] > 0)
            for k in ("total_ms", "useful_flops", "launches")}


def gemm_alone_and_overlap(trace: dict, steps: int, alone_trace: dict, alone_steps: int, peaks: dict,
                           workload: dict = None):
    """`roofline_alone` (the GEMM from the traced steps without the overlap)
    and the `overlap` summary (None when the timed steps had no pooled work)."""
    roof_alone = None
    g_alone = gemm_totals(alone_trace)
    if g_alone["total_ms"] > 0:
        a_alone = g_alone["useful_flops"] / (g_alone["total_ms"] * 1e-3) / 1e12
        sus = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
        roof_alone = {"bound": "tensor", "kernel": "gemm_tcgen05", "achieved": a_alone, "peak": sus,
                      "unit": "TFLOP/s", "frac": a_alone / sus, "peak_burst": peaks["bf16_tflops"],
                      "frac_burst": a_alone / peaks["bf16_tflops"],
                      "launches_per_step": g_alone["launches"] / alone_steps,
                      "method": "3 extra traced steps with the accumulation overlap off"}
        tr_alone = traffic_record("gemm_tcgen05", workload)
        roof_alone["traffic"] = tr_alone["dram_bytes_per_launch"] if tr_alone else None
    overlap = None
    if "accum_pool" in trace or "scatter_pool" in trace:
        def per_step(tr, name, n):
            return tr.get(name, {}).get("total_ms", 0.0) / n
        overlap = {
            "on": True,
            "gemm_ms_per_step": gemm_totals(trace)["total_ms"] / steps,
            "gemm_ms_per_step_alone": g_alone["total_ms"] / alone_steps,
            "accum_standalone_ms_per_step": per_step(trace, "accum_rownorm", steps),
            "accum_pool_rest_ms_per_step": per_step(trace, "accum_pool", steps),
            "accum_ms_per_step_alone": per_step(alone_trace, "accum_rownorm", alone_steps),
            "scatter_standalone_ms_per_step": per_step(trace, "scatter_update", steps),
            "scatter_pool_rest_ms_per_step": per_step(trace, "scatter_pool", steps),
            "scatter_ms_per_step_alone": per_step(alone_trace, "scatter_update", alone_steps),
            "method": ("the first shape group's accumulation runs on its own; each later group's is a pool "
                       "of rows taken by streaming warps inside the previous group's GEMM launches, the "
                       "rest by a pool kernel; the last group's GEMM launches carry the scatter updates "
                       "of up to two earlier groups the same way")}
    return roof_alone, overlap


def rank_barrier(world: int):
    if world > 1:
        import torch
        torch.distributed.barrier()


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def build_state(groups, device, seed_base, d3):
    """Per-group contiguous [batch, n, m] tensors; seeded Gaussian W and G,
    zero momentum (the warm-up steps fill it)."""
    import torch
    import workloads
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}
    state = []
    for gi, (r, c, b, pd, gd) in enumerate(groups):
        W = torch.empty((b, r, c), dtype=dt[pd], device=device)
        G = torch.empty((b, r, c), dtype=dt[gd], device=device)
        M = torch.zeros((b, r, c), dtype=torch.float32, device=device)
        for i in range(b):
            workloads.device_gaussian_(W[i], 0.02, seed_base + 100000 * gi + 2 * i)
            workloads.device_gaussian_(G[i], 0.01, seed_base + 100000 * gi + 2 * i + 1)
        state.append({"W": W, "G": G, "M": M, "rows": r, "cols": c, "batch": b,
                      "group": d3.Group(params=list(W.unbind(0)), grads=list(G.unbind(0)),
                                        momentum=list(M.unbind(0)))})
    return state


def cpu_baseline(state, groups, f, hp, flops_total):
    """Time the float64 oracle on one matrix per shape group (the state as it is
    now), scale by the group sizes."""
    import numpy as np
    from oracle import dion3_step as oracle_step
    t_est = 0.0
    parts = []
    for st, (r, c, b, pd, gd) in zip(state, groups):
        W = st["W"][0].float().cpu().numpy()
        M = st["M"][0].cpu().numpy()
        G = st["G"][0].float().cpu().numpy()
        t0 = time.perf_counter()
        oracle_step(W, M, G, f=f, mu=hp.mu, lr=hp.lr, eps=hp.eps, param_dtype=pd)
        dt = time.perf_counter() - t0
        t_est += dt * b
        parts.append(f"{r}x{c}: {dt:.2f} s x {b}")
    ms = t_est * 1e3
    return {"value": flops_total / (t_est * 1e12), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "ms_per_step_est": ms,
            "sample": "float64 oracle on one matrix of each shape group, scaled by group size ("
                      + "; ".join(parts) + ")"}


#: The (model, f) points of the per-model table printed with the default
#: workload (the 7B f = 1/4 point is the headline measurement itself).
PER_MODEL_POINTS = (("7b", 0.125), ("1b", 1.0), ("1b", 0.5), ("1b", 0.25))


def time_steps(state, hp, d3, device, stream, world, steps, warmup, lazy):
    """Device ms per dion3_step (or dion3_step_lazy) over every group of
    `state`, CUDA events on `stream` after `warmup` untimed steps; max over
    ranks."""
    import torch
    cg = [st_["group"] for st_ in state]
    ws = d3.alloc_workspace(d3.workspace_size(cg, hp), device=device)
    sel = [torch.empty((st_["batch"], d3.num_selected(hp.f, st_["rows"])), dtype=torch.int32, device=device)
           for st_ in state]
    scales = [torch.ones((st_["batch"], st_["rows"]), dtype=torch.float32, device=device) for st_ in state]

    def one():
        if lazy:
            d3.step_lazy(cg, hp, scales, ws, sel_idx_out=sel, stream=stream)
        else:
            d3.step(cg, hp, ws, sel_idx_out=sel, stream=stream)

    for _ in range(warmup):
        one()
    rank_barrier(world)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(device)
    rank_barrier(world)
    d3.device_status(stream)
    ms = e0.elapsed_time(e1) / steps
    del ws, sel, scales
    return max_over_ranks(ms, world, device)


def path_fractions(trace, steps, peaks):
    """The two parts of the step measured against their own roofline, from a
    launch trace of `steps` steps: the Gram-NS path (every tcgen05 GEMM launch,
    timed per Newton-Schulz chain) in useful TFLOP/s against the measured
    sustained and burst bf16 peaks, and the select/update path (the memory-bound
    kernels) in algorithmic GB/s against the measured HBM copy bandwidth."""
    gemm = [v for v in trace.values() if v["useful_flops"] > 0]
    mem = [v for v in trace.values() if v["useful_flops"] == 0]
    g_ms = sum(v["total_ms"] for v in gemm)
    g_fl = sum(v["useful_flops"] for v in gemm)
    m_ms = sum(v["total_ms"] for v in mem)
    m_b = sum(v["algo_bytes"] for v in mem)
    sus = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
    out = {}
    if g_ms > 0:
        tf = g_fl / (g_ms * 1e-3) / 1e12
        out.update({"gram_ns_ms_per_step": g_ms / steps, "gram_ns_tflops": tf,
                    "gram_ns_frac_sustained": tf / sus, "gram_ns_frac_burst": tf / peaks["bf16_tflops"]})
    if m_ms > 0:
        gbs = m_b / (m_ms * 1e-3) / 1e9
        out.update({"select_update_ms_per_step": m_ms / steps, "select_update_gbs": gbs,
                    "select_update_frac_hbm": gbs / peaks["hbm_gbs"]})
    return out


def traced_alone(state, hp, d3, stream, steps, lazy, overlap_after=True):
    """A launch trace of `steps` extra steps with the accumulation overlap off,
    so every kernel does only its own part: the GEMM launches carry no
    accumulation rows.  The overlap is set back to `overlap_after`."""
    import torch
    cg = [st_["group"] for st_ in state]
    ws = d3.alloc_workspace(d3.workspace_size(cg, hp))
    scales = [torch.ones((st_["batch"], st_["rows"]), dtype=torch.float32, device=ws.device) for st_ in state]
    d3.set_overlap(False)
    d3.trace_enable(True)
    try:
        for _ in range(steps):
            if lazy:
                d3.step_lazy(cg, hp, scales, ws, stream=stream)
            else:
                d3.step(cg, hp, ws, stream=stream)
        trace = d3.trace_collect()
    finally:
        d3.trace_enable(False)
        d3.set_overlap(overlap_after)
    d3.device_status(stream)
    del ws, scales
    return trace


def traced_fractions(state, hp, d3, stream, steps, lazy, peaks, overlap_after=True):
    """path_fractions over `steps` extra steps, each part on its own (launch
    trace on, accumulation overlap off; the step time itself is taken without
    the trace and with the overlap as configured)."""
    return path_fractions(traced_alone(state, hp, d3, stream, steps, lazy, overlap_after), steps, peaks)


def per_model_table(args, world, device, stream, d3, hp_kwargs, main_state, head_row, peak):
    """ms and useful TFLOP/s of the step for each (model, f) point: the 7B
    set (already resident) at the other f, then the 1B set, built for it; and
    the Gram-NS and select/update paths of each against their rooflines."""
    peaks, _ = load_peaks()
    rows = [head_row]
    states = {"7b": main_state}
    for model, f in PER_MODEL_POINTS:
        groups, _ = workload_groups(model)
        if model not in states:
            states[model] = build_state(groups, device, 11, d3)
        hp = d3.HParams(f=f, **hp_kwargs)
        flops = useful_flops_total(groups, f, hp_kwargs, d3)
        ms = time_steps(states[model], hp, d3, device, stream, world, args.per_model_steps, 3, args.lazy_decay)
        tflops = job_tflops(flops, world, ms)
        row = {"model": model.upper(), "f": f, "ms_per_step": ms, "useful_tflops": tflops,
               "frac_of_fp16_peak": tflops / world / peak}
        row.update(traced_fractions(states[model], hp, d3, stream, 3, args.lazy_decay, peaks,
                                    overlap_after=not args.no_overlap))
        rows.append(row)
    return rows


def run_ours(args, rank, world, device_index):
    import torch
    import matrix_orthogonalizing_optimizer_shape_gb300 as d3

    torch.cuda.set_device(device_index)
    device = torch.device("cuda", device_index)
    d3.load_library()
    d3.set_overlap(not args.no_overlap)
    groups, desc = workload_groups(args.workload, args.max_batch)
    hp_kwargs = dict(mu=0.95, lr=0.02, eps=1e-7, ns_steps=5, restart_iter=3,
                     ns_dtype=d3.BF16 if args.ns_dtype == "bf16" else d3.F16)
    hp = d3.HParams(f=args.f, **hp_kwargs)
    flops_rank = useful_flops_total(groups, args.f, hp_kwargs, d3)

    state = build_state(groups, device, 7 + 1000003 * rank, d3)
    cgroups = [s["group"] for s in state]
    ws = d3.alloc_workspace(d3.workspace_size(cgroups, hp), device=device)
    sel = [torch.empty((s["batch"], d3.num_selected(args.f, s["rows"])), dtype=torch.int32,
                       device=device) for s in state]
    stream = torch.cuda.current_stream(device)
    # Lazy decay (--lazy-decay): per-row pending factors, one [batch, rows]
    # buffer per group, starting at 1.
    scales = [torch.ones((st_["batch"], st_["rows"]), dtype=torch.float32, device=device) for st_ in state]
    # Per-neuron normalisation (--normuon): per-row second moments, one
    # [batch, rows] buffer per group, starting at 0.
    nm = d3.NormuonParams()
    vstate = [torch.zeros((st_["batch"], st_["rows"]), dtype=torch.float32, device=device) for st_ in state]

    def do_step(grps, scl, sel_out, wsp, vst=None, stream_=stream):
        if args.normuon:
            d3.step_normuon(grps, hp, nm, vst if vst is not None else vstate, wsp, sel_idx_out=sel_out,
                            stream=stream_)
        elif args.lazy_decay:
            d3.step_lazy(grps, hp, scl, wsp, sel_idx_out=sel_out, stream=stream_)
        else:
            d3.step(grps, hp, wsp, sel_idx_out=sel_out, stream=stream_)

    def barrier():
        rank_barrier(world)

    for _ in range(args.warmup):
        do_step(cgroups, scales, sel, ws)
    d3.device_status(stream)

    # Timed region: K steps, kernel times from the library trace (events per
    # memory-bound launch and per chain of GEMM launches).
    clocks = ClockSampler(device_index)
    barrier()
    torch.cuda.synchronize(device)
    clocks.start()
    d3.trace_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        do_step(cgroups, scales, sel, ws)
    ev1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clock_info = clocks.stop()
    trace = d3.trace_collect()
    d3.trace_enable(False)
    d3.device_status(stream)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, world, device)
    launches = sum(v["launches"] for v in trace.values())
    # Each part on its own (accumulation overlap off), for the path fractions
    # and the GEMM's own roofline.
    alone_steps = 3
    alone_trace = traced_alone(state, hp, d3, stream, alone_steps, args.lazy_decay,
                               overlap_after=not args.no_overlap)

    # The same step captured once in a CUDA graph and replayed K times: no
    # host launch overhead between the step's kernels (the library enqueues
    # kernels only, so a step can be captured).
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        cg_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg_, stream=side):
            do_step(cgroups, scales, sel, ws, stream_=None)   # on the capturing stream
        for _ in range(args.warmup):
            cg_.replay()
        barrier()
        torch.cuda.synchronize(device)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            cg_.replay()
        g1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
        d3.device_status(stream)
        gms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world, device)
        graph = {"value": job_tflops(flops_rank, world, gms), "unit": "TFLOP/s", "ms_per_step": gms,
                 "method": "one step captured in a CUDA graph, replayed per timed step"}
        del cg_

    # End to end: every step copies its gradients from pinned host memory and
    # reads the selected rows back, through the public API.  The CPU-GPU link
    # (about 210 GB/s measured on this machine) is the bound, so the copies are
    # pipelined with the compute: each shape group is cut into sub-batches of
    # at most `chunk` matrices; a copy stream moves them in order and the
    # compute stream steps each sub-batch (dion3_step on that sub-group) as soon
    # as its gradients have landed.  Sub-batches with the least compute go last.
    e2e = None
    if not args.no_e2e:
        chunk = args.e2e_chunk
        pieces = []  # (group index, lo, hi)
        for gi, st_ in enumerate(state):
            for lo in range(0, st_["batch"], chunk):
                pieces.append((gi, lo, min(st_["batch"], lo + chunk)))
        # least Gram-NS work per matrix last
        order = sorted(range(len(state)), key=lambda gi: -d3.useful_flops(
            d3.num_selected(args.f, state[gi]["rows"]), state[gi]["cols"], hp))
        pieces.sort(key=lambda pc: order.index(pc[0]))
        host_g = [torch.empty(st_["G"].shape, dtype=st_["G"].dtype, pin_memory=True).copy_(st_["G"])
                  for st_ in state]
        host_sel = [torch.empty(x.shape, dtype=torch.int32).pin_memory() for x in sel]
        sub_groups = []
        for (gi, lo, hi) in pieces:
            st_ = state[gi]
            sub_groups.append(d3.Group(params=[st_["W"][i] for i in range(lo, hi)],
                                       grads=[st_["G"][i] for i in range(lo, hi)],
                                       momentum=[st_["M"][i] for i in range(lo, hi)]))
        ws_e2e = d3.alloc_workspace(max(d3.workspace_size([g], hp) for g in sub_groups), device=device)
        copy_stream = torch.cuda.Stream(device)
        h2d = sum(h.numel() * h.element_size() for h in host_g)
        d2h = sum(h.numel() * h.element_size() for h in host_sel)

        def e2e_step():
            start_ev = stream.record_event()
            copy_stream.wait_event(start_ev)
            evs = []
            with torch.cuda.stream(copy_stream):
                for (gi, lo, hi) in pieces:
                    state[gi]["G"][lo:hi].copy_(host_g[gi][lo:hi], non_blocking=True)
                    evs.append(copy_stream.record_event())
            for (gi, lo, hi), ev, sg in zip(pieces, evs, sub_groups):
                stream.wait_event(ev)
                do_step([sg], [scales[gi][lo:hi]], [sel[gi][lo:hi]], ws_e2e, [vstate[gi][lo:hi]])
            for x, h in zip(sel, host_sel):
                h.copy_(x, non_blocking=True)

        e2e_step()  # warm the sub-group path
        barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
        e2e = {"value": job_tflops(flops_rank, world, ems), "unit": "TFLOP/s",
               "ms_per_step": ems, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "method": f"pinned host gradients copied on a side stream in sub-batches of <= {chunk} "
                         "matrices, each sub-batch stepped as soon as it lands; the selected row indices "
                         "read back to pinned host memory; W and M (the optimizer state) stay resident in "
                         "HBM, as in training",
               "h2d_gbs": h2d / (ems * 1e-3) / 1e9}
        del host_g, ws_e2e

    per_model = None
    if args.workload == "7b" and args.f == 0.25 and args.max_batch == 0 and not args.no_per_model \
            and not args.normuon:
        peaks0, _ = load_peaks()
        peak0 = peaks0.get("bf16_tflops_sustained") or peaks0["bf16_tflops"]
        head = {"model": "7B", "f": args.f, "ms_per_step": ms_max,
                "useful_tflops": job_tflops(flops_rank, world, ms_max),
                "frac_of_fp16_peak": job_tflops(flops_rank, world, ms_max) / world / peak0}
        head.update(path_fractions(alone_trace, alone_steps, peaks0))
        per_model = per_model_table(args, world, device, stream, d3, hp_kwargs, state, head, peak0)

    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    dom_name, dom = max(trace.items(), key=lambda kv: kv[1]["total_ms"])
    if dom["useful_flops"] > 0:
        achieved = dom["useful_flops"] / (dom["total_ms"] * 1e-3) / 1e12
        peak = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "peak_kind": f"bf16 sustained ({peak_src}); fp16 dense rate = bf16 dense rate"}
    else:
        achieved = dom["algo_bytes"] / (dom["total_ms"] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "peak_kind": f"hbm copy ({peak_src})"}
    roof["frac"] = achieved / peak
    if "accum_pool" in trace or "scatter_pool" in trace:
        roof["note"] = ("the GEMM launches also carry the streaming warps that move part of the next "
                        "shape group's accumulation and of earlier groups' scatter updates (see overlap); "
                        "roofline_alone is the GEMM on its own")
    if roof["bound"] == "tensor":
        # the same rate against the burst figure (a kernel timed on its own)
        roof["peak_burst"] = peaks["bf16_tflops"]
        roof["frac_burst"] = achieved / peaks["bf16_tflops"]
    roof["kernel"] = dom_name
    roof["launches_per_step"] = dom["launches"] / args.steps
    tr = traffic_record(dom_name, traffic_workload(args))
    # The record is the GEMM on its own; launches that also carry accumulation
    # rows move more, so their traffic is left open.
    side = "accum_pool" in trace or "scatter_pool" in trace
    roof["traffic"] = tr["dram_bytes_per_launch"] if tr and not side else None
    kernels = {}
    tot_ms = sum(v["total_ms"] for v in trace.values())
    for name, v in sorted(trace.items(), key=lambda kv: -kv[1]["total_ms"]):
        kv = {"launches_per_step": v["launches"] / args.steps,
              "ms_per_step": v["total_ms"] / args.steps, "share": v["total_ms"] / tot_ms}
        if v["useful_flops"] > 0:
            kv["tflops"] = v["useful_flops"] / (v["total_ms"] * 1e-3) / 1e12
        if v["algo_bytes"] > 0 and v["useful_flops"] == 0 and name not in ("accum_pool", "scatter_pool"):
            kv["gbs"] = v["algo_bytes"] / (v["total_ms"] * 1e-3) / 1e9
        if name == "accum_pool":
            kv["note"] = "the rows of the pooled accumulations that the GEMM launches' streaming warps left"
        if name == "scatter_pool":
            kv["note"] = "the rows of the deferred scatter updates that the GEMM launches' streaming warps left"
        kernels[name] = kv

    value = job_tflops(flops_rank, world, ms_max)
    bf16_peak = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
    # Step roofline: the GEMM phase at the sustained tensor peak plus the
    # memory-bound phase at the measured copy bandwidth (the phases are serial
    # within a group), against the measured step.
    hbm_bytes = sum(v["algo_bytes"] for v in trace.values() if v["useful_flops"] == 0) / args.steps
    t_tensor = flops_rank / (bf16_peak * 1e12) * 1e3
    t_hbm = hbm_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    step_roof = {"t_roof_ms": t_tensor + t_hbm, "tensor_part_ms": t_tensor, "hbm_part_ms": t_hbm,
                 "useful_tflop": flops_rank / 1e12, "hbm_gb": hbm_bytes / 1e9,
                 "peak_tflops": bf16_peak, "hbm_gbs": peaks["hbm_gbs"],
                 "frac": (t_tensor + t_hbm) / ms_max}
    if graph is not None:
        step_roof["frac_graph"] = (t_tensor + t_hbm) / graph["ms_per_step"]
    paths = path_fractions(alone_trace, alone_steps, peaks)
    roof_alone, overlap = gemm_alone_and_overlap(trace, args.steps, alone_trace, alone_steps, peaks,
                                                 traffic_workload(args))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.ns_dtype, "data": "synthetic",
        "config": workload_config(args, groups, desc),
        "useful_tflop_per_step_per_gpu": flops_rank / 1e12,
        "frac_of_fp16_peak": value / world / bf16_peak,
        "parallelism": f"{world} independent ranks (no collective on the data path)",
        "roofline": roof, "roofline_alone": roof_alone, "overlap": overlap,
        "step_roofline": step_roof, "paths": paths, "kernels": kernels,
        "gpu_launches": launches,
        "gpu_launches_per_step": launches / args.steps, "clocks": clock_info,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if per_model is not None:
        line["per_model"] = per_model
    if graph is not None:
        line["graph"] = graph
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(state, groups, args.f, hp, flops_rank)
    return line


# ---------------------------------------------------------------------------
# Gram-NS sweep: fp16 Gaussian X, s x L with L = s * aspect, batch of same-shape
# matrices; our four Newton-Schulz variants and cuBLAS (torch fp16 bmm)
# running the Gram schedule and standard NS as reference points.
# ---------------------------------------------------------------------------

def _cublas_gram_ns(X, hp):
    """Gram NS with torch fp16 batched matmuls (cuBLAS), same schedule."""
    import torch
    a, b, c = hp.coeffs
    Y = X / (X.float().pow(2).sum(dim=(1, 2), keepdim=True).sqrt().half() + hp.eps)
    s = Y.shape[1]
    eye = torch.eye(s, device=X.device, dtype=X.dtype).expand(Y.shape[0], s, s)
    R = torch.bmm(Y, Y.transpose(1, 2))
    Q = None
    for t in range(1, hp.ns_steps + 1):
        if t == hp.restart_iter and t > 1:
            Y = torch.bmm(Q, Y)
            R = torch.bmm(Y, Y.transpose(1, 2))
            Q = None
        Z = torch.baddbmm(torch.add(eye * a, R, alpha=b), R, R, alpha=c)
        Q = Z if Q is None else torch.bmm(Z, Q)
        if t < hp.ns_steps and t + 1 != hp.restart_iter:
            R = torch.bmm(Z, torch.bmm(R, Z))
    return torch.bmm(Q, Y)


def _cublas_standard_ns(X, hp):
    import torch
    a, b, c = hp.coeffs
    Y = X / (X.float().pow(2).sum(dim=(1, 2), keepdim=True).sqrt().half() + hp.eps)
    for _ in range(hp.ns_steps):
        A = torch.bmm(Y, Y.transpose(1, 2))
        B = torch.baddbmm(A * b, A, A, alpha=c)
        Y = torch.baddbmm(Y * a, B, Y)
    return Y


def run_sweep(args):
    import torch
    import matrix_orthogonalizing_optimizer_shape_gb300 as d3
    import workloads
    d3.load_library()
    hp = d3.HParams()
    if args.sweep_points:
        # explicit points "s x L x batch" (Gram side, long side, matrices)
        pts = []
        for item in args.sweep_points.split(","):
            s_, L_, b_ = (int(v) for v in item.lower().split("x"))
            pts.append((s_, L_ // s_, b_))
    elif args.sweep_full:
        pts = [(s, a, b) for s in workloads.SWEEP_S for a in workloads.SWEEP_ASPECT
               for b in workloads.SWEEP_BATCH]
    else:
        # one batch per (s, aspect), chosen for about 20 TFLOP of Gram-NS work
        pts = []
        for s_ in workloads.SWEEP_S:
            for a in (1, 4):
                L = s_ * a
                work = 6.0 * s_ * s_ * L + 14.0 * s_ ** 3
                b = max(1, min(64, int(2e13 // work)))
                b = max(x for x in workloads.SWEEP_BATCH if x <= b)
                pts.append((s_, a, b))
    names = {d3.NS_GRAM: "gram", d3.NS_GRAM_DENSE: "gram_dense", d3.NS_STANDARD: "standard",
             d3.NS_STANDARD_DENSE: "standard_dense"}
    only = set(v for v in args.sweep_variants.split(",") if v) if args.sweep_variants else None
    if only:
        names = {v: n for v, n in names.items() if n in only}
        if not names:
            raise SystemExit("--sweep-variants names none of gram, gram_dense, standard, standard_dense")
    rows = []
    s_ev = torch.cuda.current_stream()
    for (s_, a, b) in pts:
        L = s_ * a
        # X + O + workspace of the largest variant must fit comfortably
        need = 2 * b * s_ * L * 2 + max(d3.ns_workspace_size(v, s_, L, b, hp) for v in names)
        if need > 200e9:
            rows.append({"s": s_, "L": L, "batch": b, "skipped": "over 200 GB"})
            continue
        g = torch.Generator(device="cuda")
        g.manual_seed(s_ * 131 + a * 7 + b)
        X = torch.randn((b, s_, L), generator=g, device="cuda", dtype=torch.float32).half()
        O = torch.empty_like(X)
        row = {"s": s_, "L": L, "batch": b}
        for v, name in names.items():
            ws = d3.alloc_workspace(d3.ns_workspace_size(v, s_, L, b, hp))
            for _ in range(2):
                d3.ns_batched(v, X, O, hp, ws)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_ev)
            for _ in range(args.steps):
                d3.ns_batched(v, X, O, hp, ws)
            e1.record(s_ev)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            row[name + "_ms"] = ms
            row[name + "_tflops"] = b * d3.ns_useful_flops(v, s_, L, hp) / (ms * 1e-3) / 1e12
            del ws
        d3.device_status()
        for name, fn in (("cublas_gram", _cublas_gram_ns), ("cublas_standard", _cublas_standard_ns)):
            if only is not None and name not in only:
                continue
            for _ in range(2):
                fn(X, hp)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_ev)
            for _ in range(args.steps):
                fn(X, hp)
            e1.record(s_ev)
            torch.cuda.synchronize()
            row[name + "_ms"] = e0.elapsed_time(e1) / args.steps
        for ref in ("standard", "standard_dense", "cublas_standard", "cublas_gram"):
            if "gram_ms" in row and ref + "_ms" in row:
                row["speedup_vs_" + ref] = row[ref + "_ms"] / row["gram_ms"]
        rows.append(row)
        del X, O
        torch.cuda.empty_cache()
    peaks, src = load_peaks()
    return {"metric": "Gram-NS sweep: ms and useful TFLOP/s per variant", "unit": "TFLOP/s",
            "data": "synthetic", "dtype": "f16", "steps": args.steps,
            "peak_bf16_tflops_sustained": peaks.get("bf16_tflops_sustained"), "peak_source": src,
            "config": {"workload": "fp16 Gaussian X, s x L, T=5 restart@3 (standard NS: T=5)"},
            "points": rows}


# ---------------------------------------------------------------------------
# Reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    import numpy as np
    import workloads
    from oracle import dion3_step as oracle_step, num_selected as o_num_selected

    groups, desc = workload_groups(args.workload, args.max_batch)
    # Useful FLOPs of the Gram-NS schedule, counted with the oracle's own op log.
    from oracle import gram_newton_schulz, gram_ns_useful_flops
    log = []
    gram_newton_schulz(np.ones((2, 3)) / 6.0, steps=5, restart_iter=3, op_log=log)
    flops = 0.0
    for (r, c, b, pd, gd) in groups:
        k = o_num_selected(args.f, r)
        s, L = min(k, c), max(k, c)
        flops += b * gram_ns_useful_flops([(op[0], s, L) if op[0] != "sym" else ("sym", s)
                                           for op in log])
    samples = []
    for (r, c, b, pd, gd) in groups:
        samples.append({
            "W": workloads.gaussian((r, c), 0.02, seed=1, dtype=pd),
            "M": workloads.gaussian((r, c), 0.05, seed=2),
            "G": workloads.gaussian((r, c), 0.01, seed=3, dtype=gd)})
    # Each step runs the oracle on ONE matrix, rotating through the shape groups.
    # `value` is the oracle's useful throughput on this workload: the full set's
    # FLOPs over the full set's time as the sampled per-matrix times put it
    # (each group's latest time times its size).  `ms_per_step` is the wall time
    # a sampled step actually took; the full-set estimate is reported beside it.
    # W >= 3 warm-up steps cover every group of the model-shaped sets first.
    group_t = [None] * len(groups)
    est, walls = [], []
    for it in range(args.warmup + args.steps):
        g = it % len(groups)
        smp = samples[g]
        r, c, b, pd, gd = groups[g]
        t0 = time.perf_counter()
        W, M, _, _ = oracle_step(smp["W"], smp["M"], smp["G"], f=args.f, mu=0.95, lr=0.02,
                                 param_dtype=pd)
        dt = time.perf_counter() - t0
        group_t[g] = dt
        smp["W"], smp["M"] = W.astype(np.float32), M
        if it >= args.warmup:
            est.append(sum(t * grp[2] for t, grp in zip(group_t, groups)))
            walls.append(dt)
    full_ms = 1e3 * sum(est) / len(est)
    value = flops / (full_ms * 1e-3) / 1e12
    ms = 1e3 * sum(walls) / len(walls)
    sample = ("float64 oracle on one matrix per step, rotating through the shape groups "
              f"({', '.join(f'{r}x{c} x{b}' for (r, c, b, _, _) in groups)}); value = the full set's useful "
              "FLOPs over the sum of each group's latest per-matrix time times its size")
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_full_set_est": full_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args, groups, desc),
            "useful_tflop_per_step_per_gpu": flops / 1e12,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b", choices=["7b", "1b", "gapped", "single", "sweep"])
    ap.add_argument("--sweep-full", action="store_true",
                    help="with --workload sweep: every (s, aspect, batch) of the sweep grid")
    ap.add_argument("--sweep-points", default="",
                    help="with --workload sweep: comma-separated points SxLxBATCH (e.g. 512x4096x128)")
    ap.add_argument("--sweep-variants", default="",
                    help="with --workload sweep: comma-separated subset of gram, gram_dense, standard, "
                         "standard_dense, cublas_gram, cublas_standard (default: all)")
    ap.add_argument("--f", type=float, default=0.25)
    ap.add_argument("--lazy-decay", action="store_true",
                    help="dion3_step_lazy: the selected rows' decay is carried to the next step")
    ap.add_argument("--normuon", action="store_true",
                    help="dion3_step_normuon: per-neuron normalisation of the orthogonalised rows "
                         "(NorMuon reading; the per-model table is skipped)")
    ap.add_argument("--ns-dtype", choices=["f16", "bf16"], default="f16",
                    help="16-bit type of the Gram-NS operands (the pages use fp16)")
    ap.add_argument("--max-batch", type=int, default=0,
                    help="cap the matrices per shape group (small profiling case)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="run the shape groups without the accumulation overlap (dion3_set_overlap(0))")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=16,
                    help="matrices per pipelined sub-batch in the end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay measurement")
    ap.add_argument("--no-per-model", action="store_true",
                    help="skip the per-model table (7B at f = 1/8, 1B at f = 1, 1/2, 1/4)")
    ap.add_argument("--per-model-steps", type=int, default=10,
                    help="timed steps per point of the per-model table")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.workload == "sweep":
        if rank == 0 and args.impl == "ours":
            print(json.dumps(run_sweep(args)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
