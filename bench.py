#!/usr/bin/env python3
"""Benchmark of the fused exact-attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward pass (one launch of the sm_103a kernel through the C
ABI) over one batch of the workload; the default workload is the SD2.1 UNet
self-attention block (B=2, H=5, N=4096, d=64, no mask), on which the metric is
quoted. Inputs are seeded synthetic bf16 tensors already resident in HBM; the
timed steps rotate over enough input sets that together exceed the 129 MB L2,
so no step reads another step's inputs from L2.

Metric: attention forward TFLOP/s, counting 4 * 128 * 128 * d per 128x128
(query, key) tile of a fixed reference grid that holds at least one allowed
pair (for no mask this is 4 * Nq * Nk * d per head); the exact count of
allowed pairs is reported beside it.

One JSON line on rank 0 with: value (whole-job TFLOP/s, the K timed steps
replayed as one CUDA graph between two events on its stream), roofline of the
kernel (its average launch duration from those events, against the measured
bf16 peak; eager per-launch events beside it as a cross-check), e2e (the same
metric with every step's inputs copied in from pinned host memory and its
outputs read back inside the timed region: a stream of calls whose copies
overlap the neighbouring steps' kernels; the one-stream serial figure beside
it), cpu_baseline (the fp64 CPU oracle on a bounded sample), clocks sampled
during the timed region.

With --impl reference the line is the CPU oracle itself (the only reference
implementation: the pages ship no code), timed on the host cores.

Multi-GPU (torchrun, one process per GPU): every rank runs its own instance of
the workload (independent problems, no data-path collective); value = all
ranks' work / the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from seeded_inputs import WORKLOADS, make_qkv  # noqa: E402

METRIC = "attention fwd TFLOP/s (4·Nq·Nk·d/head) and % of GB300 bf16 tensor peak"
DEFAULT_WORKLOAD = "sd21_unet_block"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["exact_attention_69_gb300/csrc/attn_sm103.cuh",
                  "exact_attention_69_gb300/csrc/tmem_ldst.inc",
                  "exact_attention_69_gb300/csrc/attn_kernel.h"]


# ------------------------------------------------------------------ counting

def _axis_allowed(G: int, k: int, wrap: bool) -> np.ndarray:
    c = np.arange(G)[:, None]
    e = np.arange(G)[None, :]
    if wrap:
        return ((e - c + k // 2) % G) < k
    s = np.clip(c - k // 2, 0, G - k)
    return (e >= s) & (e < s + k)


def allowed_pairs_matrix(w) -> np.ndarray | None:
    """Boolean [Nq, Nk] allowed-pair matrix for masked workloads (None: no mask)."""
    if w.mask == "none":
        return None
    if w.mask == "causal":
        return np.tril(np.ones((w.Nq, w.Nk), dtype=bool))
    wraps = w.wrap_axes if w.wrap_axes is not None else (w.mask == "wrap",) * len(w.grid)
    m = np.ones((1, 1), dtype=bool)
    for G, wrap in zip(w.grid, wraps):  # row-major tokens: the first axis is the slowest
        m = np.kron(m, _axis_allowed(G, w.window, wrap))
    return m.astype(bool)


def count_flops(w):
    """(tile-rule flops, exact allowed-pair flops) for the whole workload."""
    per_pair = 4.0 * w.d * w.B * w.H
    m = allowed_pairs_matrix(w)
    if m is None:
        f = per_pair * w.Nq * w.Nk
        return f, f
    nq, nk = -(-w.Nq // 128), -(-w.Nk // 128)
    pad = np.zeros((nq * 128, nk * 128), dtype=bool)
    pad[:w.Nq, :w.Nk] = m
    tiles = pad.reshape(nq, 128, nk, 128).any(axis=(1, 3)).sum()
    return per_pair * 128 * 128 * float(tiles), per_pair * float(m.sum())


def host_cpu_model() -> str:
    """The host CPU as the OS names it (model name, or the Arm implementer and
    part numbers), with the machine type."""
    import platform
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        for key in ("model name", "Model name", "Hardware"):
            for ln in info:
                if ln.split(":")[0].strip() == key:
                    name = ln.split(":", 1)[1].strip()
                    break
            if name:
                break
        if not name:
            impl = next((ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU implementer")), "")
            part = next((ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU part")), "")
            if impl or part:
                name = f"implementer {impl} part {part}"
    except OSError:
        pass
    return f"{name or platform.processor() or 'unknown'} ({platform.machine()})"


def percentile(xs, q):
    """q-th percentile (0..100) of a list, linear between order statistics."""
    ys = sorted(xs)
    if not ys:
        return None
    pos = (len(ys) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


# ------------------------------------------------------------------ multi-rank

def max_over_ranks(ms: float, dist_mod, device) -> float:
    """The slowest rank's time (every rank gets it); `ms` itself on one rank."""
    if dist_mod is None or not dist_mod.is_available() or not dist_mod.is_initialized():
        return ms
    if dist_mod.get_world_size() == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, steps: int, ms_total: float) -> float:
    """All ranks' work (each rank runs its own instance: weak scaling) over the
    slowest rank's time."""
    return world * flops_per_rank_step * steps / (ms_total * 1e-3) / 1e12


def rank_seed(w, rank: int) -> int:
    """Each rank draws its own instance of the workload."""
    return w.seed + 1000 * rank


# ------------------------------------------------------------------ environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_sha") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons in a background thread."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [p for (t, p) in self.samples if t0 - 0.05 <= t <= t1 + 0.05]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            window = "nearest sample to a timed region shorter than the 100 ms sampling period"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ CPU oracle

class OracleSampler:
    """The fp64 oracle on bounded row samples of workload w: inputs prepared
    and the cost per row measured once; each run() times one random sample of
    rows spread over every (batch, head)."""

    def __init__(self, w):
        import oracle
        from seeded_inputs import make_workload, to_f64
        self.oracle = oracle
        q, k, v = make_workload(w)
        self.qf, self.kf, self.vf = to_f64(q), to_f64(k), to_f64(v)
        self.total = w.B * w.H * w.Nq
        self.kw = dict(scale=w.scale, mask_kind=w.mask, window=w.window, grid=w.grid,
                       wrap=w.wrap_axes if w.wrap_axes is not None else False)
        n = min(self.total, 64)
        rows = np.sort(np.random.default_rng(7).choice(self.total, size=n, replace=False))
        t = time.perf_counter()
        oracle.attention_rows(self.qf, self.kf, self.vf, rows, **self.kw)
        self.per_row = max((time.perf_counter() - t) / n, 1e-7)
        self.threads = oracle.max_threads()

    def run(self, target_s: float, seed_rows: int, min_rows: int = 1):
        """(seconds, rows) of one sample sized to take about target_s."""
        n = int(min(self.total, max(min_rows, target_s / self.per_row)))
        rows = np.sort(np.random.default_rng(seed_rows).choice(self.total, size=n, replace=False))
        t = time.perf_counter()
        self.oracle.attention_rows(self.qf, self.kf, self.vf, rows, **self.kw)
        return time.perf_counter() - t, n


def oracle_sample(w, target_s: float, seed_rows: int = 7):
    """Time the fp64 oracle on a bounded row sample of workload w.

    Returns (seconds, rows, total_rows, threads)."""
    smp = OracleSampler(w)
    dt, n = smp.run(target_s, seed_rows, min_rows=64)
    return dt, n, smp.total, smp.threads


def reference_arm(args, w):
    """--impl reference: the CPU oracle timed on the host cores, one bounded
    row sample of the workload per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    flops_tile, _ = count_flops(w)
    # each step a bounded sample; the whole run (warm-up and timed steps)
    # stays within ATTN_REF_TOTAL_S seconds of oracle work
    n_all = max(1, args.warmup + args.steps)
    per_step_target = min(float(os.environ.get("ATTN_REF_STEP_S", "3.0")),
                          float(os.environ.get("ATTN_REF_TOTAL_S", "90")) / n_all)
    smp = OracleSampler(w)
    times, rows_done = [], 0
    total_rows, threads = smp.total, smp.threads
    for i in range(n_all):
        dt, n = smp.run(per_step_target, seed_rows=100 + i)
        if i >= args.warmup:
            times.append(dt)
            rows_done += n
    total_s = sum(times)
    value = flops_tile * (rows_done / total_rows) / total_s / 1e12
    sample = (f"about {rows_done // max(args.steps, 1)} of the {total_rows} query rows per step "
              f"(random rows of every head), {args.steps} timed steps, fp64, "
              f"{threads} OpenMP threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, rotating_sets=None),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "cpu_model": host_cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, rotating_sets):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
           "mask": w.mask, "scale": w.scale, "sigma": w.sigma, "seed": w.seed,
           "flop_rule": "4*128*128*d per 128x128 reference tile holding an allowed pair"}
    if w.mask in ("clamp", "wrap"):
        cfg.update({"window": w.window, "grid": list(w.grid), "dilation": w.dilation})
        if w.wrap_axes is not None:
            cfg["wrap_axes"] = list(w.wrap_axes)
    if rotating_sets is not None:
        cfg["l2"] = (f"inputs larger than L2: {rotating_sets} rotating input sets "
                     f"(> {L2_BYTES // 2**20} MiB in total), no explicit flush")
        cfg["launch"] = "K timed steps captured in one CUDA graph, replayed once"
    return cfg


# ------------------------------------------------------------------ GPU arm

def ours_arm(args, w):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from exact_attention_69_gb300 import build as _build
    _build.build()
    import exact_attention_69_gb300 as E

    flops_tile, flops_exact = count_flops(w)
    set_bytes = 2 * (2 * w.B * w.H * w.Nq * w.d + 2 * w.B * w.H * w.Nk * w.d) + 4 * w.B * w.H * w.Nq
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes))
    q, k, v = make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.sigma, rank_seed(w, rank))
    sets = []
    for i in range(n_sets):
        # distinct device buffers per set (same values): no step hits L2 from the last
        sets.append((q.to(dev), k.to(dev), v.to(dev),
                     torch.empty(w.B, w.H, w.Nq, w.d, dtype=torch.bfloat16, device=dev),
                     torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device=dev)))
    stream = torch.cuda.current_stream(dev)
    kw = dict(scale=w.scale, mask=w.mask, window=w.window, grid=w.grid, wrap_axes=w.wrap_axes)

    def step(i, events=None):
        qq, kk, vv, oo, ll = sets[i % n_sets]
        E.attn_fwd(qq, kk, vv, out=oo, lse=ll, events=events, **kw)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    code, detail = E.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} {detail} after warm-up")

    # The K timed steps are captured once into a CUDA graph and replayed, so the
    # device runs them back to back with no host launch gaps; the graph holds
    # exactly K launches of the kernel (the workspace, if any, was allocated
    # during the warm-up).
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(args.steps):
            step(i)
    torch.cuda.synchronize()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()).start() if rank == 0 else None
    if sampler:
        time.sleep(0.3)  # let nvidia-smi start sampling
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    with torch.cuda.stream(cap):  # replay() launches on the current stream
        t_start.record(cap)
        graph.replay()
        t_stop.record(cap)
    torch.cuda.synchronize()
    h1 = time.time()
    if world > 1:
        dist.barrier()
    clocks = sampler.summary(h0, h1) if sampler else None
    if sampler:
        sampler.stop()
    code, detail = E.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} {detail} in the timed region")
    ms_total = t_start.elapsed_time(t_stop)
    # cross-check: eager launches, each bracketed by events on its stream
    n_eager = max(3, min(args.steps, 50))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_eager)]
    for i in range(n_eager):
        step(i, events=kev[i])
    torch.cuda.synchronize()
    k_ms = [a.elapsed_time(b) for a, b in kev]
    ms_total = max_over_ranks(ms_total, dist if world > 1 else None, dev)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(world, flops_tile, args.steps, ms_total)

    # End to end through the public API: pinned host inputs in, host outputs back,
    # every step. A stream of independent calls: step i's inputs are copied in on
    # one stream, its kernel runs on a second, its outputs are copied out on a
    # third, with three device buffer sets, so the copies of steps i + 1 and i - 1
    # overlap the kernel of step i and the next step's copy in never waits for
    # the read-back of the step before (events order each buffer's reuse). The same
    # steps one after the other on one stream are reported as serial_value.
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    n_bufs = 3
    bufs = [sets[i] for i in range(min(n_bufs, n_sets))]
    while len(bufs) < n_bufs:  # filled by each step's own copy in before its kernel reads it
        bufs.append(tuple(torch.empty_like(t) for t in sets[0]))
    oh = [torch.empty(bufs[0][3].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(n_bufs)]
    lh = [torch.empty(bufs[0][4].shape, dtype=torch.float32, pin_memory=True) for _ in range(n_bufs)]
    e_steps = max(3, min(args.steps, 200))
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(n_bufs)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_bufs)]
    ev_out = [torch.cuda.Event() for _ in range(n_bufs)]
    used = [False] * n_bufs

    def e2e_step(i):
        b = i % n_bufs
        qd, kd, vd, od, ld = bufs[b]
        if used[b]:  # buffer b's last kernel and read-back are done
            s_in.wait_event(ev_out[b])
        used[b] = True
        with torch.cuda.stream(s_in):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        E.attn_fwd(qd, kd, vd, out=od, lse=ld, stream=s_cmp, **kw)
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            oh[b].copy_(od, non_blocking=True)
            lh[b].copy_(ld, non_blocking=True)
        ev_out[b].record(s_out)

    def e2e_serial_step():
        qd, kd, vd, od, ld = bufs[0]
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        E.attn_fwd(qd, kd, vd, out=od, lse=ld, **kw)
        oh[0].copy_(od, non_blocking=True)
        lh[0].copy_(ld, non_blocking=True)

    def timed(run, start_stream, end_stream):
        for i in range(3):
            run(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(start_stream)
        end_stream.wait_stream(start_stream)
        for i in range(e_steps):
            run(i)
        e1.record(end_stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dist if world > 1 else None, dev)

    s_out.wait_stream(stream)
    s_in.wait_stream(stream)
    e_ms = timed(e2e_step, s_in, s_out)
    e_ms_serial = timed(lambda i: e2e_serial_step(), stream, stream)
    code, detail = E.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} {detail} in the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh[0].numel() * oh[0].element_size() + lh[0].numel() * lh[0].element_size()
    # Both runs move every step's bytes; the faster is the end-to-end figure (short
    # steps are bound by the host's issue rate, which the three-stream form raises).
    piped = whole_job_tflops(world, flops_tile, e_steps, e_ms)
    serial = whole_job_tflops(world, flops_tile, e_steps, e_ms_serial)
    e2e = {"value": max(piped, serial), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
           "mode": "pipelined" if piped >= serial else "serial",
           "pipelined_value": piped, "pipelined_ms_per_step": e_ms / e_steps,
           "pipeline": "3 streams, 3 device buffer sets: copies of steps i+1 and i-1 overlap the kernel of step i",
           "serial_value": serial, "serial_ms_per_step": e_ms_serial / e_steps}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    k_avg_ms = ms_step  # the graph holds only this kernel: average launch duration
    achieved = flops_tile / (k_avg_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                "peak_source": f"{peak_src} bf16 burst (cuBLAS 8192^3)",
                "frac_of_sustained": achieved / float(peaks["bf16_tflops_sustained"]),
                "kernel_ms_avg": k_avg_ms,
                "kernel_ms_eager_avg": sum(k_ms) / len(k_ms), "kernel_ms_eager_min": min(k_ms),
                "kernel_ms_eager_p10": percentile(k_ms, 10), "kernel_ms_eager_p50": percentile(k_ms, 50),
                "kernel_ms_eager_p90": percentile(k_ms, 90),
                "exact_pairs_tflops": flops_exact / (k_avg_ms * 1e-3) / 1e12,
                "hbm_gbs_compulsory": set_bytes / (k_avg_ms * 1e-3) / 1e9}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        dt, n, total, threads = oracle_sample(w, float(os.environ.get("ATTN_CPU_S", "12")))
        cpu = {"value": flops_tile * (n / total) / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle", "cpu_model": host_cpu_model(),
               "sample": f"{n} of {total} query rows (random, every head) in {dt:.1f} s, fp64"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(w, n_sets),
        "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e,
        "gpu_launches": args.steps, "impl": "ours",
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w)
    return ours_arm(args, w)


if __name__ == "__main__":
    sys.exit(main())
