#!/usr/bin/env python3
"""Benchmark: int4 decode GEMV achieved HBM bandwidth on one GB300 (and N replicas).

One step = one pass of the decode projection set of an 8B-class transformer at
M = 1, group 128 (qo_proj 4096x4096, gate_up_proj 14336x4096, down_proj
4096x14336, LM head 128256x4096), each projection one q4gemv_run call through
the C ABI.  The metric is the bytes those four GEMVs must move (codes + scales
+ zero points + x + y) divided by the step time; the per-GEMV microseconds per
call are reported beside it.  The 0.5B-class set (seven projections, group 32)
is timed in the detail.

Timing method (after the harness lessons of cera's wgpu_gemv_bench.rs and the
Refractometer page):
  * the K timed steps are back-to-back launches on one stream, captured once in
    a CUDA graph and replayed, bracketed by CUDA events on that stream with a
    device synchronise (and a barrier across ranks) on both sides;
  * that timed region of exactly K steps is repeated (at least --samples times
    and for at least --sample-seconds); the value is the median region, with
    p10 / p90 beside it (the Refractometer's median and p10-p90 over samples;
    cera's "medians of several runs");
  * every step uses the next of several weight replicas whose total is several
    times the 129 MB L2, so each step streams its weights from HBM;
  * W untimed warm-up steps run first;
  * per-projection microseconds come from separate graphs of back-to-back
    launches (median of --samples replays, with t(2n)/t(n) as the ITERS check);
  * by default the GEMVs are launched overlapped (programmatic dependent
    launch: a kernel streams its weights while the previous one finishes and
    waits for it before reading x); --overlap 0 serialises them;
  * SM clocks and throttle reasons are sampled with nvidia-smi during the
    timed regions.

`--impl reference` times the CPU oracle (the plain C restatement of the
method) on the host cores instead; there is no other reference implementation
of this path.  Under torchrun each rank runs an independent replica of the
workload on its own GPU (the GEMV has no exchange step); rank 0 prints one
JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
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

import synth  # noqa: E402

HEADLINE = synth.DECODE_8B   # the timed step: its projections at M = 1

METRIC = "int4 GEMV achieved HBM GB/s (% of GB300 peak) and µs/call at M=1, 1 GPU"
UNIT = "GB/s"
WORKLOAD = ("decode projection set of an 8B-class transformer, M=1, group=128 (qo_proj 4096x4096, "
            "gate_up_proj 14336x4096, down_proj 4096x14336, lm_head 128256x4096)")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu capture of
# the instance below on the LM-head shape (see profiles/); None once the kernel changes.
DOMINANT_KERNEL = ("q4gemv_stream_kernel<K=4096, g=128, RG=4, U=8, ASYM> (32-row blocks, 3 ring slots, "
                   "1 CTA per SM)")
DOMINANT_TRAFFIC_BYTES = 272_976_128 + 3_917_056


def algorithmic_bytes(M, N, K, group, symmetric=False):
    """Bytes one GEMV must move once: codes + fp16 scales + 4-bit zeros + x + y."""
    nb = K // group
    w = N * (K // 2) + N * nb * 2 + (0 if symmetric else N * ((nb + 1) // 2))
    return w + M * K * 4 + M * N * 4


def step_bytes(shapes, M=1, group=32):
    return sum(algorithmic_bytes(M, N, K, group) for _, N, K in shapes)


# ----------------------------------------------------------------- ranks

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_over_ranks(dist, value: float, op: str, device=None) -> float:
    """MAX or SUM of a per-rank float over all ranks (identity on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"--loop-ms={self.interval}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(self.interval / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        window = [p for ts, p in rows if (t0 is None or ts >= t0) and (t1 is None or ts <= t1)]
        use = window if window else [p for ts, p in rows]
        sm = [float(p[1]) for p in use if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in use:
            for name, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(window)}


def smi_index(local_rank: int) -> int:
    """nvidia-smi index of this rank's GPU (CUDA_VISIBLE_DEVICES may remap it)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    if local_rank < len(vis) and vis[local_rank].strip().isdigit():
        return int(vis[local_rank])
    return local_rank


# ----------------------------------------------------------------- peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- graph events

class GraphEvents:
    """Timing events that can be recorded as nodes of a captured CUDA graph."""

    def __init__(self, torch):
        self.torch = torch
        self.rt = None
        try:
            torch.cuda.Event(enable_timing=True, external=True)
            self.mode = "torch"
        except TypeError:
            self.mode = "cudart"
            self.rt = ctypes.CDLL("libcudart.so.13")
            self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
            self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                         ctypes.c_uint]
            self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float),
                                                     ctypes.c_void_p, ctypes.c_void_p]

    def new(self):
        if self.mode == "torch":
            return self.torch.cuda.Event(enable_timing=True, external=True)
        ev = ctypes.c_void_p()
        assert self.rt.cudaEventCreate(ctypes.byref(ev)) == 0
        return ev

    def record(self, ev, stream):
        if self.mode == "torch":
            ev.record(stream)
        else:
            assert self.rt.cudaEventRecordWithFlags(ev, stream.cuda_stream, 1) == 0

    def elapsed_ms(self, a, b):
        if self.mode == "torch":
            return a.elapsed_time(b)
        ms = ctypes.c_float()
        assert self.rt.cudaEventElapsedTime(ctypes.byref(ms), a, b) == 0
        return ms.value


# ----------------------------------------------------------------- GPU arm

def make_weights(shapes, group, scale, seed=2024):
    return [synth.q4_weights(seed + i, N, K, group, scale_range=scale, tag=name)
            for i, (name, N, K) in enumerate(shapes)]


class StepSet:
    """One decode projection set on the device: its host weights (for the oracle legs),
    rotating device replicas whose total exceeds the L2 several times (every step streams
    its weights from HBM), one x and one y per projection (M = 1)."""

    def __init__(self, torch, spec, rotate_bytes, seed=2024):
        self.shapes = spec["shapes"]
        self.group = spec["group"]
        self.ws = make_weights(self.shapes, self.group, spec["scale"], seed)
        self.replica_bytes = sum(w.nbytes for w in self.ws)
        self.replicas = max(2, -(-rotate_bytes // self.replica_bytes))
        self.reps = [[(to_dev(torch, w.codes), to_dev(torch, w.scales), to_dev(torch, w.zeros)) for w in self.ws]
                     for _ in range(self.replicas)]
        self.xs_host = [synth.activations_f32(77 + i, 1, K) for i, (_, _, K) in enumerate(self.shapes)]
        self.xs = [to_dev(torch, x) for x in self.xs_host]
        self.ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in self.shapes]
        self.bytes_per_step = step_bytes(self.shapes, 1, self.group)

    def step(self, q4, r, stream):
        for p, (name, N, K) in enumerate(self.shapes):
            c, sc, z = self.reps[r][p]
            q4.q4gemv_run(c, sc, z, self.xs[p], self.ys[p], 1, N, K, self.group, stream=stream)


def to_dev(torch, a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def capture_steps(torch, stream, step, n, offset, replicas):
    """A CUDA graph of n back-to-back steps over the rotating replicas."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            step((offset + i) % replicas)
    return g


def quantiles(v):
    t = sorted(v)
    q = lambda f: t[min(len(t) - 1, max(0, int(round(f * (len(t) - 1)))))]
    return {"median": statistics.median(t), "p10": q(0.1), "p90": q(0.9), "min": t[0], "max": t[-1],
            "mean": statistics.fmean(t)}


def timed_regions(torch, stream, dist, run_region, min_samples, min_seconds, max_samples=20000):
    """Repeat the timed region (exactly K steps, issued by run_region) at least min_samples
    times and for at least min_seconds: each sample is bracketed by a barrier and a device
    synchronise on both sides and timed by CUDA events on the launching stream; its time
    is the maximum over ranks.  Returns the per-sample milliseconds and the host-clock
    window they span."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    t0 = time.monotonic()
    while len(ms) < max_samples and (len(ms) < min_samples or time.monotonic() - t0 < min_seconds):
        barrier(dist)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            run_region()
            end.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        ms.append(reduce_over_ranks(dist, start.elapsed_time(end), "max", device="cuda"))
    return ms, t0, time.monotonic()


def run_gpu(args, rank, world, local_rank):
    import torch
    import gemm_decode_gb300 as q4

    torch.cuda.set_device(local_rank)
    dist = dist_init(world, "nccl")
    q4.lib()
    q4.q4gemv_set_overlapped_launch(bool(args.overlap))
    S = StepSet(torch, HEADLINE, args.rotate_bytes)
    shapes, group, replicas = S.shapes, S.group, S.replicas
    stream = torch.cuda.Stream()
    LM = len(shapes) - 1   # the dominant launch: the LM head

    # eager pass over every replica (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for r in range(replicas):
            S.step(q4, r, stream)
    torch.cuda.synchronize()

    # the timed region: exactly K steps, as replays of a graph of `chunk` steps (plus a tail)
    chunk = max(1, min(args.steps, max(replicas, args.graph_steps)))
    full, tail = divmod(args.steps, chunk)
    step = lambda r: S.step(q4, r, stream)
    g_main = capture_steps(torch, stream, step, chunk, 0, replicas)
    g_tail = capture_steps(torch, stream, step, tail, full * chunk, replicas) if tail else None

    def region():
        for _ in range(full):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()

    # warm-up: exactly W steps
    if args.warmup:
        wn = min(args.warmup, chunk)
        g_warm = capture_steps(torch, stream, step, wn, 0, replicas)
        wfull, wtail = divmod(args.warmup, wn)
        g_wtail = capture_steps(torch, stream, step, wtail, 0, replicas) if wtail else None
        with torch.cuda.stream(stream):
            for _ in range(wfull):
                g_warm.replay()
            if g_wtail is not None:
                g_wtail.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(smi_index(local_rank)).start()
    time.sleep(0.3)
    samples_ms, t0, t1 = timed_regions(torch, stream, dist, region, args.samples, args.sample_seconds)
    clocks = sampler.stop(t0, t1)
    qs = quantiles(samples_ms)
    ms_region = qs["median"]
    total_bytes = S.bytes_per_step * args.steps * world
    value = total_bytes / (ms_region * 1e-3) / 1e9
    gbs_of = lambda ms: round(total_bytes / (ms * 1e-3) / 1e9, 2)

    # per-GEMV microseconds per call: for each projection, a graph of back-to-back launches
    # over the rotating replicas (no event nodes between launches), 25 timed replays
    n_pp = max(replicas, min(args.steps, 200), 40)
    per_proj = [_time_back_to_back(torch, q4, stream, [r[p] for r in S.reps], S.xs[p], S.ys[p], 1, N, K, group,
                                   n_pp, samples=args.samples)
                for p, (name, N, K) in enumerate(shapes)]

    # the dominant launch inside the step: event nodes around every LM-head launch of a
    # separate (untimed) graph of steps; the nodes break the launch overlap around them
    ev = GraphEvents(torch)
    n_ev = min(chunk, 50)
    events = [(ev.new(), ev.new()) for _ in range(n_ev)]
    g_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ev, stream=stream):
        for i in range(n_ev):
            for p, (name, N, K) in enumerate(shapes):
                c, sc, z = S.reps[i % replicas][p]
                if p == LM:
                    ev.record(events[i][0], stream)
                q4.q4gemv_run(c, sc, z, S.xs[p], S.ys[p], 1, N, K, group, stream=stream)
                if p == LM:
                    ev.record(events[i][1], stream)
    with torch.cuda.stream(stream):
        g_ev.replay()
        g_ev.replay()
    torch.cuda.synchronize()
    lm_in_step_us = statistics.median(ev.elapsed_ms(a, b) * 1e3 for a, b in events)

    peak, peak_src = load_peaks()
    lm_bytes = algorithmic_bytes(1, shapes[LM][1], shapes[LM][2], group)
    lm_us = per_proj[LM]["us"]
    achieved = lm_bytes / (lm_us * 1e-6) / 1e9
    in_step = lm_bytes / (lm_in_step_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": DOMINANT_KERNEL + f" on {shapes[LM][0]} {shapes[LM][1]}x{shapes[LM][2]}",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": args.traffic_bytes if args.traffic_bytes is not None else DOMINANT_TRAFFIC_BYTES,
                "algorithmic_bytes_per_launch": lm_bytes,
                "duration_us": round(lm_us, 3),
                "duration_p10_p90": [round(per_proj[LM]["p10"], 3), round(per_proj[LM]["p90"], 3)],
                "duration_source": "CUDA events on the launching stream around a graph of back-to-back "
                                   "LM-head launches (rotating replicas, cold L2, overlapped launch), "
                                   f"median of {args.samples} replays, right after the timed regions",
                "in_step": {"us": round(lm_in_step_us, 3), "achieved": round(in_step, 1),
                            "frac": round(in_step / peak, 4),
                            "how": "event nodes around every LM-head launch of a separate graph of steps; "
                                   "they break the launch overlap and add a bubble, so this figure is "
                                   "conservative"}}

    # ---- end to end: pinned host x in, pinned host y out, through the same API ----
    e2e = run_e2e(args, torch, q4, shapes, group, S.reps, S.xs_host, replicas, stream, dist)

    us_per_call = {name: round(st["us"], 3) for (name, N, K), st in zip(shapes, per_proj)}
    detail = {"projections": [
        {"name": name, "N": N, "K": K, "us_per_call": round(st["us"], 3),
         "gbs": round(algorithmic_bytes(1, N, K, group) / (st["us"] * 1e-6) / 1e9, 1),
         "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
         "t2n_over_tn": round(st["t2n_over_tn"], 3), "launches_per_sample": st["n"]}
        for (name, N, K), st in zip(shapes, per_proj)],
        "weight_replicas": replicas, "replica_bytes": S.replica_bytes, "graph_steps": chunk,
        "event_mode": ev.mode,
        "us_per_call_note": f"per projection: a graph of back-to-back launches over the rotating replicas, "
                            f"{args.samples} timed replays (median; p10, p90, min) and t(2n)/t(n) from two "
                            f"replays"}
    if args.controls and rank == 0:
        try:   # a detail figure: its failure is recorded, the measured step stands
            detail["grouped_step"] = run_grouped_step(args, torch, q4, shapes, group, S.reps, S.xs, replicas, stream)
        except Exception as e:   # noqa: BLE001
            detail["grouped_step"] = {"error": f"{type(e).__name__}: {e}"}
        detail["decode_05b"] = run_decode_05b(args, torch, q4, stream)
        detail["controls"] = run_controls(args, torch, q4)
        detail["prefill_tensor_core"] = run_prefill(args, torch, q4)
        detail["decode_8b"] = run_decode_8b(args, torch, q4)
        detail["q4_0_format"] = run_q40(args, torch, q4)
        try:   # a detail figure: its failure is recorded, the measured step stands
            detail["q8_0_format"] = run_q80(args, torch, q4)
        except Exception as e:   # noqa: BLE001
            detail["q8_0_format"] = {"error": f"{type(e).__name__}: {e}"}

    probe = detail.get("controls", {}).get("vec4_read_probe_1GiB", {}).get("gbs")
    if probe:   # the same kernel's rate against this GPU's own streaming read (the vec4 probe)
        roofline["frac_of_read_probe"] = round(roofline["achieved"] / probe, 4)
        roofline["read_probe_gbs"] = probe
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_region / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights (fp16 scales, u4 zeros), f32 x/accumulate/y",
        "data": "synthetic (seeded; codes/zeros uniform 0..15, scales fp16 U[0.001,0.01], x N(0,1))",
        "config": {"workload": WORKLOAD, "M": 1, "group": group,
                   "shapes": [[n, N, K] for n, N, K in shapes],
                   "bytes_per_step": S.bytes_per_step,
                   "l2_policy": f"inputs larger than L2: {replicas} rotating weight replicas "
                                f"({replicas * S.replica_bytes / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": ("overlapped: programmatic dependent launch, each GEMV waits for the "
                              "previous kernel before reading x" if args.overlap else "serialised")},
        "timing": {"samples": len(samples_ms), "statistic": "median over timed regions of exactly K steps",
                   "ms_per_region": {k: round(v, 6) for k, v in qs.items()},
                   "value_p10_p90": [gbs_of(qs["p90"]), gbs_of(qs["p10"])],
                   "seconds_sampled": round(t1 - t0, 3)},
        "us_per_call": us_per_call,
        "clocks": clocks, "e2e": e2e, "gpu_launches": len(shapes) * args.steps,
        "gpu_launches_note": "per timed region (each sample is one region of K steps)",
        "roofline": roofline, "pct_of_8TBs_nominal": round(value / NOMINAL_HBM_GBS, 4),
        "detail": detail,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, S.ws, S.xs_host, shapes, group,
                                              gpu_outputs=[y.cpu().numpy() for y in S.ys])
    return result, dist


def run_decode_05b(args, torch, q4, stream):
    """The decode projection set of a 0.5B-class model at M = 1, group 32 (seven GEMVs per
    step): the step as a graph of back-to-back launches, each projection's microseconds per
    call, the step with stacked q|k|v and gate|up and with the RMSNorm / SwiGLU fusions, and
    the step as two grouped calls."""
    S = StepSet(torch, synth.DECODE_05B, args.rotate_bytes)
    shapes, group, replicas = S.shapes, S.group, S.replicas
    n = max(replicas, min(args.steps, 400), 100)
    st = _time_launches(torch, stream, lambda i: S.step(q4, i % replicas, stream), n, samples=args.samples)
    per_proj = [_time_back_to_back(torch, q4, stream, [r[p] for r in S.reps], S.xs[p], S.ys[p], 1, N, K, group,
                                   max(replicas, 200), samples=args.samples)
                for p, (name, N, K) in enumerate(shapes)]
    out = {"workload": "decode projection set of a 0.5B-class transformer, M=1, group=32",
           "shapes": [[nm, N, K] for nm, N, K in shapes], "bytes_per_step": S.bytes_per_step,
           "us_per_step": round(st["us"], 3), "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3),
                                                                 round(st["min"], 3)],
           "gbs": round(S.bytes_per_step / st["us"] / 1e3, 1), "t2n_over_tn": round(st["t2n_over_tn"], 3),
           "steps_per_sample": n, "samples": args.samples,
           "projections": [{"name": name, "N": N, "K": K, "us_per_call": round(p["us"], 3),
                            "gbs": round(algorithmic_bytes(1, N, K, group) / (p["us"] * 1e-6) / 1e9, 1),
                            "us_p10_p90_min": [round(p["p10"], 3), round(p["p90"], 3), round(p["min"], 3)],
                            "t2n_over_tn": round(p["t2n_over_tn"], 3)}
                           for (name, N, K), p in zip(shapes, per_proj)]}
    out["fused_projections_step"] = run_fused_step(args, torch, q4, shapes, group, S.reps, S.xs, replicas, stream)
    try:   # a detail figure: its failure is recorded, the measured step stands
        out["grouped_step"] = run_grouped_step(args, torch, q4, shapes, group, S.reps, S.xs, replicas, stream)
    except Exception as e:   # noqa: BLE001
        out["grouped_step"] = {"error": f"{type(e).__name__}: {e}"}
    del S
    torch.cuda.empty_cache()
    return out


def run_e2e(args, torch, q4, shapes, group, reps, xs_host, replicas, stream, dist):
    """The step end to end from pinned host memory, three ways, each a CUDA graph of K steps:
      mapped          -- q4gemv_run reads x from and writes y to pinned host memory directly
                         (device-addressable over NVLink-C2C; the transfers happen inside the
                         kernels' loads and stores, no copy nodes);
      copy            -- one host->device copy of every x and one device->host copy of every y
                         per step around the seven launches on device buffers;
      x_copy_y_mapped -- the x copy, then launches that store y straight into pinned host memory.
    `value` is the fastest; all are reported, and their y must agree bit for bit."""
    xcat_h = torch.from_numpy(np.concatenate([x.reshape(-1) for x in xs_host])).pin_memory()
    xcat_d = torch.empty_like(xcat_h, device="cuda")
    ntot = sum(N for _, N, _ in shapes)
    ycat_d = torch.empty(ntot, dtype=torch.float32, device="cuda")
    ycat_h = torch.empty(ntot, dtype=torch.float32).pin_memory()
    ycat_m = torch.empty(ntot, dtype=torch.float32).pin_memory()
    xoff, yoff = [], []
    o = 0
    for _, _, K in shapes:
        xoff.append(o)
        o += K
    o = 0
    for _, N, _ in shapes:
        yoff.append(o)
        o += N

    def step_copy(r):
        xcat_d.copy_(xcat_h, non_blocking=True)
        for p, (name, N, K) in enumerate(shapes):
            c, sc, z = reps[r][p]
            q4.q4gemv_run(c, sc, z, xcat_d[xoff[p]:xoff[p] + K], ycat_d[yoff[p]:yoff[p] + N],
                          1, N, K, group, stream=stream)
        ycat_h.copy_(ycat_d, non_blocking=True)

    def step_mapped(r):
        for p, (name, N, K) in enumerate(shapes):
            c, sc, z = reps[r][p]
            q4.q4gemv_run(c, sc, z, xcat_h[xoff[p]:xoff[p] + K], ycat_m[yoff[p]:yoff[p] + N],
                          1, N, K, group, stream=stream)

    ycat_y = torch.empty(ntot, dtype=torch.float32).pin_memory()

    def step_x_copy_y_mapped(r):
        xcat_d.copy_(xcat_h, non_blocking=True)
        for p, (name, N, K) in enumerate(shapes):
            c, sc, z = reps[r][p]
            q4.q4gemv_run(c, sc, z, xcat_d[xoff[p]:xoff[p] + K], ycat_y[yoff[p]:yoff[p] + N],
                          1, N, K, group, stream=stream)

    n = args.steps
    bytes_step = step_bytes(shapes, 1, group)

    def timed(step):
        with torch.cuda.stream(stream):
            for i in range(min(args.warmup, 8) + 1):
                step(i % replicas)
        torch.cuda.synchronize()
        chunk = min(n, max(replicas, args.graph_steps))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(chunk):
                step(i % replicas)
        full, tail = divmod(n, chunk)
        gt = None
        if tail:
            gt = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gt, stream=stream):
                for i in range(tail):
                    step((full * chunk + i) % replicas)
        def region():
            for _ in range(full):
                g.replay()
            if gt is not None:
                gt.replay()

        # the median of several timed regions of exactly K steps (max over ranks each)
        ms, _, _ = timed_regions(torch, stream, dist, region, max(5, args.samples // 5), 0.0)
        return statistics.median(ms)

    world = dist.get_world_size() if dist is not None else 1
    ms_copy = timed(step_copy)
    ms_mapped = timed(step_mapped)
    ms_ymap = timed(step_x_copy_y_mapped)
    # all ways compute the same y (same kernels, same inputs): compare on replica 0
    with torch.cuda.stream(stream):
        step_copy(0)
        step_mapped(0)
        step_x_copy_y_mapped(0)
    torch.cuda.synchronize()
    same = bool(torch.equal(ycat_h, ycat_m)) and bool(torch.equal(ycat_h, ycat_y))

    # the same through eager Python calls (no graph): what a plain script pays per step
    neager = min(n, 200)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(neager):
            step_mapped(i % replicas)
    torch.cuda.synchronize()
    eager_s = time.perf_counter() - t0

    def gbs(ms):
        return round(bytes_step * n * world / (ms * 1e-3) / 1e9, 2)

    nl = len(shapes)
    hows = {"copy": f"CUDA graph of K steps: pinned-host x -> device copy, {nl} x q4gemv_run, y -> pinned host copy",
            "mapped": f"CUDA graph of K steps; {nl} x q4gemv_run reading x from and writing y to pinned host memory "
                      "(NVLink-C2C, no copy nodes)",
            "x_copy_y_mapped": f"CUDA graph of K steps: pinned-host x -> device copy, {nl} x q4gemv_run writing y "
                               "straight to pinned host memory (NVLink-C2C)"}
    times = {"copy": ms_copy, "mapped": ms_mapped, "x_copy_y_mapped": ms_ymap}
    best = min(times, key=times.get) if same else "copy"
    ms = times[best]
    return {"value": gbs(ms), "unit": UNIT,
            "h2d_bytes_per_step": int(xcat_h.numel() * 4),
            "d2h_bytes_per_step": int(ycat_h.numel() * 4),
            "ms_per_step": round(ms / n, 6),
            "how": hows[best],
            "mapped": {"value": gbs(ms_mapped), "ms_per_step": round(ms_mapped / n, 6)},
            "x_copy_y_mapped": {"value": gbs(ms_ymap), "ms_per_step": round(ms_ymap / n, 6)},
            "copy": {"value": gbs(ms_copy), "ms_per_step": round(ms_copy / n, 6)},
            "mapped_equals_copy": same,
            "eager_python_calls": {"value": round(bytes_step * neager / eager_s / 1e9, 2),
                                   "ms_per_step": round(eager_s * 1e3 / neager, 4),
                                   "steps": neager, "how": "mapped"}}


def run_controls(args, torch, q4):
    """The f32 control and the read probe, timed ABBA with the int4 LM-head GEMV."""
    N, K, g = 151936, 896, 32
    w = synth.q4_weights(11, N, K, g)
    W = synth.dense_f32(11, N, K)
    x = synth.activations_f32(11, 1, K)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()
    nrep_q4 = 8
    q4w = [(dev(w.codes), dev(w.scales), dev(w.zeros)) for _ in range(nrep_q4)]
    Wd = [dev(W) for _ in range(2)]   # 2 x 545 MB: each launch reads the other copy
    xd = dev(x)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    probe_bytes = 1 << 30
    pbuf = torch.zeros(probe_bytes // 4, dtype=torch.float32, device="cuda")
    partial = torch.zeros(8192, dtype=torch.float32, device="cuda")

    def t_q4(n):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(n):
            c, sc, z = q4w[i % nrep_q4]
            q4.q4gemv_run(c, sc, z, xd, y, 1, N, K, g)
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n

    def t_f32(n):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(n):
            q4.f32gemv_run(Wd[i % 2], xd, y, 1, N, K)
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n

    def t_probe(n):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(n):
            q4.vec4_read_probe_run(pbuf, probe_bytes, partial)
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n

    t_q4(4), t_f32(2), t_probe(2)
    a1, b1 = t_q4(40), t_f32(10)
    b2, a2 = t_f32(10), t_q4(40)
    p = t_probe(10)
    qa = statistics.fmean([a1, a2])
    fb = statistics.fmean([b1, b2])
    return {
        "order": "ABBA (A = int4 GEMV, B = f32 GEMV), rotating replicas, cold L2",
        "int4_lm_head": {"us": round(qa * 1e3, 2),
                         "gbs": round(algorithmic_bytes(1, N, K, g) / (qa * 1e-3) / 1e9, 1)},
        "f32_lm_head": {"us": round(fb * 1e3, 2),
                        "gbs": round((N * K * 4 + K * 4 + N * 4) / (fb * 1e-3) / 1e9, 1)},
        "vec4_read_probe_1GiB": {"us": round(p * 1e3, 2), "gbs": round(probe_bytes / (p * 1e-3) / 1e9, 1)},
    }


def load_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


def run_prefill(args, torch, q4):
    """The tensor-core int4 matmul on the prefill shapes: TFLOP/s against the
    measured dense bf16 peak (2*M*N*K flops per call), from a CUDA graph of back-to-back
    calls on one weight copy (median of replays, as the GEMV figures)."""
    out = []
    burst, sustained, src = load_bf16_peak()
    stream = torch.cuda.Stream()
    for name, M, N, K in synth.PREFILL["shapes"]:
        w = synth.q4_weights(7, N, K, 32, tag=name)
        a = synth.activations_bf16(7, M, K)
        dev = lambda x: None if x is None else torch.from_numpy(
            np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
        cw, sw, zw, ad = dev(w.codes), dev(w.scales), dev(w.zeros), dev(a)
        c = torch.empty((M, N), dtype=torch.float32, device="cuda")
        n_it = 20 if M * N * K > 1e10 else 200
        st = _time_launches(torch, stream, lambda i: q4.q4gemm_run(cw, sw, zw, ad, c, M, N, K, 32, stream=stream),
                            n_it, samples=5)
        assert q4.q4gemv_device_status() == q4.Q4_OK
        us = st["us"]
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out.append({"name": name, "M": M, "N": N, "K": K, "us": round(us, 2), "tflops": round(tf, 1),
                    "frac_of_bf16_peak": round(tf / burst, 4), "peak": burst, "peak_source": src,
                    "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
                    "t2n_over_tn": round(st["t2n_over_tn"], 3),
                    "note": "a graph of back-to-back calls on one weight copy (W fits in L2), median of 5 replays; "
                            + ("overlapped launch" if getattr(args, "overlap", 1) else "serialised launch")})
    return out


# ----------------------------------------------------------------- CPU oracle

def oracle_step(ws, xs_host, shapes, group, threads, row_fraction=1.0):
    """One step of the oracle: every projection (or its first rows), all threads."""
    import oracle
    outs = []
    done_bytes = 0
    for w, x, (name, N, K) in zip(ws, xs_host, shapes):
        n = max(1, int(round(N * row_fraction)))
        codes, scales = w.codes[:n], w.scales[:n]
        zeros = None if w.zeros is None else w.zeros[:n]
        if threads == 1:
            y, b = oracle.q4_gemv(codes, scales, zeros, x, group)
        else:
            y, b = oracle.q4_gemv_threaded(codes, scales, zeros, x, group, threads)
        outs.append((y, b))
        done_bytes += algorithmic_bytes(1, n, K, group)
    return outs, done_bytes


def cpu_baseline(args, ws, xs_host, shapes, group, gpu_outputs=None):
    """The oracle timed on the host cores: full steps over all cores (row slices), then a
    bounded sample on one core (the first rows of every projection); the all-core run's
    outputs gate the GPU run's parity on every row."""
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    outs, nbytes = oracle_step(ws, xs_host, shapes, group, threads)
    steps = 1
    while time.perf_counter() - t0 < args.cpu_seconds:
        oracle_step(ws, xs_host, shapes, group, threads)
        steps += 1
    dt = time.perf_counter() - t0
    res = {"value": round(nbytes * steps / dt / 1e9, 4), "unit": UNIT, "cores": threads,
           "kind": "oracle",
           "sample": f"{steps} full step(s) of the projection set (all rows), "
                     f"{threads} threads over row slices, {dt:.1f} s wall"}
    # one core: the first rows of every projection, sized to about --cpu-seconds
    t0 = time.perf_counter()
    _, b_probe = oracle_step(ws, xs_host, shapes, group, 1, 0.002)
    est = (time.perf_counter() - t0) / 0.002
    frac = min(1.0, max(0.002, args.cpu_seconds / max(est, 1e-9)))
    t0 = time.perf_counter()
    _, b1 = oracle_step(ws, xs_host, shapes, group, 1, frac)
    dt1 = time.perf_counter() - t0
    res["one_core"] = {"value": round(b1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                       "sample": f"the first {frac * 100:.2f}% of the rows of every projection on one thread, "
                                 f"{dt1:.1f} s wall"}
    if gpu_outputs is not None:
        worst = 0.0
        for (y_ref, bound), y in zip(outs, gpu_outputs):
            err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
            worst = max(worst, float(np.max(err / (1e-3 * bound + 1e-6))))
        res["parity_gate"] = {"max_err_over_bound": round(worst, 6), "ok": worst <= 1.0,
                              "rows": "every row of every projection of the step"}
    return res


def run_reference(args, rank, world):
    """--impl reference: the oracle as it stands, on the host cores.  Each step is the
    oracle over the first rows of every projection (a fraction sized so that all steps
    take about --ref-seconds).  With many steps (at least four per core) they are shared
    out over one worker thread per core, each running whole steps on one core, so that no
    step pays for starting threads; with few, each step runs over all cores (row slices)."""
    if rank != 0:
        return None
    from concurrent.futures import ThreadPoolExecutor
    shapes = HEADLINE["shapes"]
    group = HEADLINE["group"]
    ws = make_weights(shapes, group, HEADLINE["scale"])
    xs_host = [synth.activations_f32(77 + i, 1, K) for i, (_, _, K) in enumerate(shapes)]
    threads = os.cpu_count() or 1
    across = args.steps >= 4 * threads
    per_step_threads = 1 if across else threads
    t0 = time.perf_counter()
    oracle_step(ws, xs_host, shapes, group, per_step_threads, 0.01)
    est_full = (time.perf_counter() - t0) / 0.01          # one full step as it will run
    budget = args.ref_seconds * (threads if across else 1) / max(1, args.steps + args.warmup)
    frac = min(1.0, budget / max(est_full, 1e-9))

    def run_steps(count):
        done = 0
        for _ in range(count):
            done += oracle_step(ws, xs_host, shapes, group, per_step_threads, frac)[1]
        return done

    if across:
        def share(total):
            return [total // threads + (1 if t < total % threads else 0) for t in range(threads)]

        with ThreadPoolExecutor(max_workers=threads) as pool:
            list(pool.map(run_steps, share(args.warmup)))
            t0 = time.perf_counter()
            nbytes = sum(pool.map(run_steps, share(args.steps)))
            dt = time.perf_counter() - t0
        how = f"on one core; the {args.steps} steps shared out over {threads} worker threads"
    else:
        run_steps(args.warmup)
        t0 = time.perf_counter()
        nbytes = run_steps(args.steps)
        dt = time.perf_counter() - t0
        how = f"over {threads} threads (row slices)"
    value = nbytes / dt / 1e9
    sample = f"each step: the first {frac * 100:.2f}% of the rows of every projection, {how}"
    return {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int4 weights, f32 x/y, f64 accumulate", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "group": group,
                       "shapes": [[n, N, K] for n, N, K in shapes]},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--samples", type=int, default=25,
                   help="timed regions of K steps (at least), and replays per microsecond figure")
    p.add_argument("--sample-seconds", type=float, default=2.0,
                   help="keep repeating the timed region for at least this long (clock samples)")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--graph-steps", type=int, default=400,
                   help="steps per captured CUDA graph (replayed to reach --steps)")
    p.add_argument("--rotate-bytes", type=int, default=6 * L2_BYTES,
                   help="total bytes of rotating weight replicas")
    p.add_argument("--cpu-seconds", type=float, default=3.0)
    p.add_argument("--ref-seconds", type=float, default=90.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--controls", type=int, default=1)
    p.add_argument("--profile", choices=["none", "lm_head", "lm_head_fused", "lm_head_8b", "down_8b", "tc_m16",
                                         "tc_lm05_m8", "tc_down8b_m8", "f32_lm_head", "gemm_ffn", "gemm_gate",
                                         "q80_lm_head_m4", "q80_lm_head_8b"],
                   default="none",
                   help="launch one kernel a few times on a small case and exit (for ncu)")
    p.add_argument("--sweep", action="store_true",
                   help="time every cell of the shape sweep instead of the decode step")
    p.add_argument("--sweep-parts", default="q4,f32,probe",
                   help="comma-separated parts of --sweep: q4 (int4 GEMV cells), f32 (control), probe (read sizes)")
    p.add_argument("--sweep-out", default=None,
                   help="JSON-lines checkpoint for --sweep: cells already in the file are not re-timed")
    p.add_argument("--overlap", type=int, default=1,
                   help="1: q4gemv_set_overlapped_launch(1) (programmatic dependent launch); 0: serialised")
    p.add_argument("--event-stride", type=int, default=25,
                   help="bracket the LM head of every n-th timed step with event nodes")
    p.add_argument("--traffic-bytes", type=float, default=None,
                   help="ncu dram bytes per launch of the dominant kernel, when measured")
    args = p.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        p.error("--steps must be >= 1 and --warmup >= 0")
    return args


PROFILE_CASES = {
    # name: (N, K, group, M); 4 rotating replicas keep each launch's weights out of L2
    "lm_head": (151936, 896, 32, 1),
    "lm_head_8b": (128256, 4096, 128, 1),
    "down_8b": (4096, 14336, 128, 1),
    "tc_m16": (32768, 4096, 128, 16),      # tensor-core GEMV, 256-row tiles, K split over clusters of 2
    "tc_lm05_m8": (151936, 896, 32, 8),    # tensor-core GEMV, 256-row tiles (two MMAs per CTA)
    "tc_down8b_m8": (4096, 14336, 128, 8), # tensor-core GEMV, K split over 8-CTA clusters
}


def run_profile_case(args):
    """A handful of launches of one kernel on a small case, for ncu captures:
    4 warm-up launches over 4 weight replicas, then 3 more."""
    import torch
    import gemm_decode_gb300 as q4
    dev = lambda a: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()
    if args.profile.startswith("gemm_"):
        name, M, N, K = synth.PREFILL["shapes"][1 if args.profile == "gemm_ffn" else 0]
        w = synth.q4_weights(7, N, K, 32, tag=name)
        a = dev(synth.activations_bf16(7, M, K))
        c = torch.empty((M, N), dtype=torch.float32, device="cuda")
        cw, sw, zw = dev(w.codes), dev(w.scales), dev(w.zeros)
        for _ in range(4):
            q4.q4gemm_run(cw, sw, zw, a, c, M, N, K, 32)
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.profile, "launches": 4}))
        return
    if args.profile.startswith("q80_"):
        N, K, M = (151936, 896, 4) if args.profile == "q80_lm_head_m4" else (128256, 4096, 1)
        reps = [dev(synth.q80_blocks(5 + i, N, K)) for i in range(2)]
        x = dev(synth.activations_f32(5, M, K))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for i in range(7):
            q4.q8_0_gemv_run(reps[i % 2], x, y, M, N, K)
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.profile, "launches": 7}))
        return
    if args.profile == "f32_lm_head":
        N, K = 151936, 896
        Ws = [dev(synth.dense_f32(3, N, K)) for _ in range(2)]
        x = dev(synth.activations_f32(3, 1, K))
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        for i in range(7):
            q4.f32gemv_run(Ws[i % 2], x, y, 1, N, K)
    elif args.profile == "lm_head_fused":
        # the LM head through q4gemv_fused_run with the RMSNorm prologue
        N, K, g, M = PROFILE_CASES["lm_head"]
        w = synth.q4_weights(5, N, K, g)
        reps = [(dev(w.codes), dev(w.scales), dev(w.zeros)) for _ in range(4)]
        x = dev(synth.activations_f32(5, M, K))
        gamma = dev(np.ones(K, np.float32))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for i in range(7):
            c, sc, z = reps[i % 4]
            q4.q4gemv_fused_run(c, sc, z, x, gamma, 1e-6, y, M, N, K, g)
    else:
        N, K, g, M = PROFILE_CASES[args.profile]
        w = synth.q4_weights(5, N, K, g)
        reps = [(dev(w.codes), dev(w.scales), dev(w.zeros)) for _ in range(4)]
        x = dev(synth.activations_f32(5, M, K))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for i in range(7):
            c, sc, z = reps[i % 4]
            q4.q4gemv_run(c, sc, z, x, y, M, N, K, g)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "launches": 7}))


def _device_q4(torch, gen, N, K, g, symmetric, scale):
    """Packed weights drawn on the device (timing inputs only; parity is the tests' job)."""
    nb = K // g
    c = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=gen)
    sc = torch.empty((N, nb), dtype=torch.float16, device="cuda").uniform_(*scale, generator=gen).view(torch.int16)
    z = None if symmetric else torch.randint(0, 256, (N, (nb + 1) // 2), dtype=torch.uint8, device="cuda",
                                             generator=gen)
    return c, sc, z


def _time_launches(torch, stream, launch, n, samples=5):
    """Microseconds per call of launch(i) from a CUDA graph of n back-to-back calls
    (i = 0 .. n-1): two eager calls, one untimed replay, then `samples` replays each
    between events on the launching stream (median, p10, p90, min), and one event pair
    around two replays (t(2n) / t(n), which is 2 when the per-call time has no fixed
    overhead in it)."""
    with torch.cuda.stream(stream):
        for i in range(2):
            launch(i)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(n):
            launch(i)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(samples + 1)]
    with torch.cuda.stream(stream):
        gr.replay()
        for i in range(samples):
            ev[i][0].record(stream)
            gr.replay()
            ev[i][1].record(stream)
        ev[samples][0].record(stream)
        gr.replay()
        gr.replay()
        ev[samples][1].record(stream)
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) * 1e3 / n for a, b in ev[:samples])
    t2 = ev[samples][0].elapsed_time(ev[samples][1]) * 1e3 / n
    med = statistics.median(t)
    q = lambda f: t[min(len(t) - 1, max(0, int(round(f * (len(t) - 1)))))]
    return {"us": med, "p10": q(0.1), "p90": q(0.9), "min": t[0], "samples": samples, "n": n,
            "t2n_over_tn": t2 / med}


def _time_back_to_back(torch, q4, stream, reps, x, y, M, N, K, g, n, samples=5):
    """Microseconds per q4gemv_run call from a CUDA graph of n back-to-back launches
    over the weight replicas (see _time_launches)."""
    nrep = len(reps)
    return _time_launches(torch, stream,
                          lambda i: q4.q4gemv_run(*reps[i % nrep], x, y, M, N, K, g, stream=stream), n, samples)


def run_fused_step(args, torch, q4, shapes, group, reps, xs, replicas, stream):
    """The decode step with q|k|v and gate|up stacked along N (the weight rows of
    projections that share x, concatenated): 4 launches per step instead of 7, the
    same weight bytes.  A CUDA graph of back-to-back steps over the replicas."""
    names = [n for n, _, _ in shapes]
    groups = [["q_proj", "k_proj", "v_proj"], ["gate_proj", "up_proj"], ["down_proj"], ["lm_head"]]
    idx = [[names.index(n) for n in gr] for gr in groups]
    fshapes, freps = [], []
    for gi in idx:
        fshapes.append(("+".join(names[i] for i in gi), sum(shapes[i][1] for i in gi), shapes[gi[0]][2]))
    for r in range(replicas):
        fr = []
        for gi in idx:
            parts = [reps[r][i] for i in gi]
            if len(parts) == 1:
                fr.append(parts[0])
                continue
            z = None if parts[0][2] is None else torch.cat([p[2] for p in parts])
            fr.append((torch.cat([p[0] for p in parts]), torch.cat([p[1] for p in parts]), z))
        freps.append(fr)
    fxs = [xs[gi[0]] for gi in idx]
    fys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in fshapes]

    def step(r):
        for p, (name, N, K) in enumerate(fshapes):
            c, sc, z = freps[r][p]
            q4.q4gemv_run(c, sc, z, fxs[p], fys[p], 1, N, K, group, stream=stream)

    n = max(replicas, min(args.steps, 400), 100)
    st = _time_launches(torch, stream, lambda i: step(i % replicas), n, samples=args.samples)
    us = st["us"]
    byts = step_bytes(fshapes, 1, group)
    out = {"launches_per_step": len(fshapes), "shapes": [[nm, N, K] for nm, N, K in fshapes],
           "us_per_step": round(us, 3), "gbs": round(byts / us / 1e3, 1), "bytes_per_step": byts,
           "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
           "t2n_over_tn": round(st["t2n_over_tn"], 3), "samples": st["samples"], "steps_per_sample": n}

    # the same four launches with the RMSNorm prologue fused into q|k|v, gate|up and the
    # LM head, and the SwiGLU combine into gate|up (its rows read as interleaved gate / up
    # pairs); down reads the combined activations gate|up leaves
    K0 = fshapes[0][2]
    gammas = [torch.from_numpy(np.random.default_rng(60 + i).uniform(0.5, 1.5, K0).astype(np.float32)).cuda()
              for i in range(3)]
    N_gu = fshapes[1][1]
    h = torch.empty((1, N_gu // 2), dtype=torch.float32, device="cuda")
    assert fshapes[2][2] == N_gu // 2

    def step_fused(r):
        (nq, Nq, Kq), (ng, Ng, Kg), (nd, Nd, Kd), (nl, Nl, Kl) = fshapes
        c, sc, z = freps[r][0]
        q4.q4gemv_fused_run(c, sc, z, fxs[0], gammas[0], 1e-6, fys[0], 1, Nq, Kq, group, stream=stream)
        c, sc, z = freps[r][1]
        q4.q4gemv_fused_run(c, sc, z, fxs[1], gammas[1], 1e-6, h, 1, Ng, Kg, group,
                            epilogue=q4.Q4_EPILOGUE_SWIGLU, stream=stream)
        c, sc, z = freps[r][2]
        q4.q4gemv_run(c, sc, z, h, fys[2], 1, Nd, Kd, group, stream=stream)
        c, sc, z = freps[r][3]
        q4.q4gemv_fused_run(c, sc, z, fxs[3], gammas[2], 1e-6, fys[3], 1, Nl, Kl, group, stream=stream)

    st2 = _time_launches(torch, stream, lambda i: step_fused(i % replicas), n, samples=args.samples)
    us2 = st2["us"]
    byts2 = byts - 4 * (N_gu // 2) + 3 * 4 * K0   # gate|up writes N/2 outputs; three gamma vectors
    # each launch of the fused step alone, back to back over the replicas
    (nq, Nq, Kq), (ng, Ng, Kg), (nd, Nd, Kd), (nl, Nl, Kl) = fshapes
    nb = max(replicas, 200)
    per_launch = {
        nq + " (RMSNorm)": _time_launches(torch, stream, lambda i: q4.q4gemv_fused_run(
            *freps[i % replicas][0], fxs[0], gammas[0], 1e-6, fys[0], 1, Nq, Kq, group, stream=stream), nb)["us"],
        ng + " (RMSNorm, SwiGLU)": _time_launches(torch, stream, lambda i: q4.q4gemv_fused_run(
            *freps[i % replicas][1], fxs[1], gammas[1], 1e-6, h, 1, Ng, Kg, group,
            epilogue=q4.Q4_EPILOGUE_SWIGLU, stream=stream), nb)["us"],
        nl + " (RMSNorm)": _time_launches(torch, stream, lambda i: q4.q4gemv_fused_run(
            *freps[i % replicas][3], fxs[3], gammas[2], 1e-6, fys[3], 1, Nl, Kl, group, stream=stream), nb)["us"],
    }
    per_launch_plain = {
        nm: _time_launches(torch, stream, lambda i, p=p, N=N, K=K: q4.q4gemv_run(
            *freps[i % replicas][p], fxs[p], fys[p], 1, N, K, group, stream=stream), nb)["us"]
        for p, (nm, N, K) in enumerate(fshapes) if p != 2}
    out["with_rmsnorm_swiglu"] = {
        "us_per_step": round(us2, 3), "gbs": round(byts2 / us2 / 1e3, 1), "bytes_per_step": byts2,
        "launches_per_step": 4,
        "us_per_launch_back_to_back": {k: round(v, 3) for k, v in per_launch.items()},
        "us_per_launch_plain": {k: round(v, 3) for k, v in per_launch_plain.items()},
        "what": "q4gemv_fused_run: RMSNorm prologue on q|k|v, gate|up and the LM head, SwiGLU epilogue on "
                "gate|up (its output feeds down); the separate norm and activation launches this replaces "
                "are not in the plain step"}
    return out


def run_grouped_step(args, torch, q4, shapes, group, reps, xs, replicas, stream):
    """The projections of a step, each with its own x and y as in the timed step, issued
    through q4gemv_grouped_run, one call per K: the matrices of one K as one streamed
    launch in which each has CTAs of its own (0.5B set: q, k, v, gate, up and the LM head
    at K = 896, down alone; 8B set: qo, gate_up and the LM head at K = 4096, down alone).
    A CUDA graph of back-to-back steps over the replicas; the outputs are checked against
    the separate calls' within the GEMV tolerance by the tests, not here."""
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in shapes]
    byK = {}
    for p, (_, N, K) in enumerate(shapes):
        byK.setdefault(K, []).append(p)

    def step(r):
        for K, ps in byK.items():
            q4.q4gemv_grouped_run([(*reps[r][p], xs[p], ys[p], shapes[p][1]) for p in ps], K, group, stream=stream)

    n = max(replicas, min(args.steps, 400), 100)
    st = _time_launches(torch, stream, lambda i: step(i % replicas), n, samples=args.samples)
    us = st["us"]
    byts = step_bytes(shapes, 1, group)
    return {"calls_per_step": len(byK), "groups": {str(K): [shapes[p][0] for p in ps] for K, ps in byK.items()},
            "us_per_step": round(us, 3), "gbs": round(byts / us / 1e3, 1), "bytes_per_step": byts,
            "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
            "t2n_over_tn": round(st["t2n_over_tn"], 3), "samples": st["samples"], "steps_per_sample": n}


def run_q40(args, torch, q4):
    """The second format (Q4_0 blocks, 18 bytes per 32 weights: 0.5625 B per weight):
    microseconds per q4_0_gemv_run call and GB/s from back-to-back launches over rotating
    replicas, next to q4gemv_run on the symmetric group-32 layout of the same shape."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(40)
    stream = torch.cuda.Stream()
    out = []
    for name, N, K, M in [("lm_head", 151936, 896, 1), ("qo_proj", 4096, 4096, 1), ("down_proj", 896, 4864, 1),
                          ("lm_head", 151936, 896, 4)]:
        nblk = K // 32
        wbytes = N * nblk * 18
        nrep = int(min(64, max(2, -(-6 * L2_BYTES // wbytes))))
        reps = []
        for _ in range(nrep):
            b = torch.randint(0, 256, (N, nblk, 18), dtype=torch.uint8, device="cuda", generator=gen)
            d = torch.empty((N, nblk), dtype=torch.float16, device="cuda").uniform_(0.005, 0.02, generator=gen)
            b[:, :, 0:2] = d.view(torch.uint8).view(N, nblk, 2)
            reps.append(b)
        x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=gen)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        st = _time_launches(torch, stream, lambda i: q4.q4_0_gemv_run(reps[i % nrep], x, y, M, N, K, stream=stream),
                            max(nrep, 100))
        byts = wbytes + 4 * M * K + 4 * M * N
        out.append({"name": name, "M": M, "N": N, "K": K, "us_per_call": round(st["us"], 3),
                    "gbs": round(byts / st["us"] / 1e3, 1), "t2n_over_tn": round(st["t2n_over_tn"], 3)})
        del reps
        torch.cuda.empty_cache()
    return {"kernel": "streamed kernel's Q4_0 instances (M = 1, long matrices: whole 18-byte blocks by bulk copy, "
                      "codes read as five 32-bit words shifted to the 2-byte offset), else the general kernel's "
                      "(nine 16-bit loads per block)", "cells": out}


def run_q80(args, torch, q4):
    """The third format (Q8_0 blocks, 34 bytes per 32 weights: 1.0625 B per weight):
    microseconds per q8_0_gemv_run call and GB/s from back-to-back launches over rotating
    replicas (cold)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(80)
    stream = torch.cuda.Stream()
    out = []
    for name, N, K, M in [("lm_head", 151936, 896, 1), ("qo_proj", 4096, 4096, 1), ("lm_head_8b", 128256, 4096, 1),
                          ("down_proj", 896, 4864, 1), ("lm_head", 151936, 896, 4)]:
        nblk = K // 32
        wbytes = N * nblk * 34
        nrep = int(min(64, max(2, -(-6 * L2_BYTES // wbytes))))
        reps = []
        for _ in range(nrep):
            b = torch.randint(0, 256, (N, nblk, 34), dtype=torch.uint8, device="cuda", generator=gen)
            d = torch.empty((N, nblk), dtype=torch.float16, device="cuda").uniform_(*synth.SCALE_Q80, generator=gen)
            b[:, :, 0:2] = d.view(torch.uint8).view(N, nblk, 2)
            reps.append(b)
        x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=gen)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        st = _time_launches(torch, stream, lambda i: q4.q8_0_gemv_run(reps[i % nrep], x, y, M, N, K, stream=stream),
                            max(nrep, 100))
        byts = wbytes + 4 * M * K + 4 * M * N
        out.append({"name": name, "M": M, "N": N, "K": K, "us_per_call": round(st["us"], 3),
                    "gbs": round(byts / st["us"] / 1e3, 1), "t2n_over_tn": round(st["t2n_over_tn"], 3)})
        del reps
        torch.cuda.empty_cache()
    return {"kernel": "streamed kernel's Q8_0 instances (M = 1, long matrices: whole 34-byte blocks by bulk copy, "
                      "codes read as nine 32-bit words shifted to the 2-byte offset, dp4a on the byte planes of x), "
                      "else a CUDA-core kernel (8 codes per lane, 2-4 weight rows per warp sharing each x load, one scale multiply per 8 codes)", "cells": out}


def run_decode_8b(args, torch, q4):
    """The 8B-class decode shapes (g = 128, M in 1, 2, 4, 8): microseconds per call and
    GB/s from back-to-back launches over rotating replicas (cold in HBM)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(8)
    stream = torch.cuda.Stream()
    g = synth.DECODE_8B["group"]
    out = []
    for name, N, K in synth.DECODE_8B["shapes"]:
        wbytes = N * K // 2 + N * (K // g) * 2 + N * ((K // g + 1) // 2)
        nrep = int(max(2, -(-6 * L2_BYTES // wbytes)))
        reps = [_device_q4(torch, gen, N, K, g, False, synth.DECODE_8B["scale"]) for _ in range(nrep)]
        for M in synth.DECODE_8B["Ms"]:
            x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=gen)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            n = int(max(nrep, min(200, 20000 / max(2.0, wbytes / 5e3))))
            st = _time_back_to_back(torch, q4, stream, reps, x, y, M, N, K, g, n)
            us = st["us"]
            out.append({"name": name, "M": M, "N": N, "K": K, "us_per_call": round(us, 3),
                        "gbs": round(algorithmic_bytes(M, N, K, g) / us / 1e3, 1),
                        "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)]})
        del reps
        torch.cuda.empty_cache()
    return out


def sweep_key(cell):
    kind = cell.get("kind", "q4")
    if kind == "f32":
        return ("f32", cell["M"], cell["N"], cell["K"])
    if kind == "probe":
        return ("probe", cell["bytes"])
    return (cell["M"], cell["N"], cell["K"], cell["group"], cell["symmetric"])


def load_sweep_checkpoint(path):
    """Cells of an earlier --sweep run (one JSON object per line), keyed by
    (M, N, K, group, symmetric) for int4 cells, ("f32", M, N, K) for the f32 control
    and ("probe", bytes) for the read probe; a missing file or path None gives none.  A line cut
    short by an interrupted run is ignored."""
    done = {}
    if not path or not os.path.exists(path):
        return done
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            try:
                c = json.loads(line)
            except json.JSONDecodeError:
                continue
            done[sweep_key(c)] = c
    return done


def run_sweep(args):
    """Every cell of the shape sweep: the int4 GEMV over (M, K, N, group, symmetric),
    the f32 control over (M, K, N), and the vec4 read probe over buffer sizes 16 KiB,
    32 KiB, ... 4 GiB (--sweep-parts picks among "q4", "f32", "probe").  Microseconds per
    call and achieved GB/s, from a CUDA graph of back-to-back launches; the GEMVs rotate
    over weight replicas (cold in HBM where the replicas exceed twice the L2), the probe
    re-reads one buffer (so sizes below the L2 show its read rate, the knee).  Inputs are
    drawn on the device (timing only; parity is the tests' job)."""
    import torch
    import gemm_decode_gb300 as q4
    q4.lib()
    q4.q4gemv_set_overlapped_launch(bool(args.overlap))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    stream = torch.cuda.Stream()
    peak, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    device = {"name": props.name, "sms": props.multi_processor_count,
              "l2_bytes": getattr(props, "L2_cache_size", None)}
    # checkpoint: cells already in --sweep-out (JSON lines) are kept and not re-timed
    done = load_sweep_checkpoint(args.sweep_out)
    out = open(args.sweep_out, "a") if args.sweep_out else None
    cells = []
    sw = synth.SWEEP
    parts = set(args.sweep_parts.split(","))

    def emit(cell):
        cells.append(cell)
        if out is not None:
            out.write(json.dumps(cell) + "\n")
            out.flush()

    for K in (sw["Ks"] if "q4" in parts else ()):
        for N in sw["Ns"]:
            for g in sw["groups"]:
                nb = K // g
                zrow = (nb + 1) // 2
                for sym in sw["symmetric"]:
                    wbytes = N * K // 2 + N * nb * 2 + (0 if sym else N * zrow)
                    todo = [M for M in sw["Ms"] if (M, N, K, g, sym) not in done]
                    cells += [done[(M, N, K, g, sym)] for M in sw["Ms"] if (M, N, K, g, sym) in done]
                    if not todo:
                        continue
                    nrep = int(min(256, max(2, -(-6 * L2_BYTES // wbytes))))
                    reps = [_device_q4(torch, gen, N, K, g, sym, sw["scale"]) for _ in range(nrep)]
                    for M in todo:
                        x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=gen)
                        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                        est_us = max(2.0, wbytes / 5e3)
                        n = int(max(nrep, min(400, 20000 / est_us)))
                        st = _time_back_to_back(torch, q4, stream, reps, x, y, M, N, K, g, n)
                        us = st["us"]
                        byts = algorithmic_bytes(M, N, K, g, symmetric=sym)
                        gbs = byts / us / 1e3
                        cell = {"M": M, "N": N, "K": K, "group": g, "symmetric": sym,
                                "us_per_call": round(us, 3), "gbs": round(gbs, 1),
                                "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
                                "t2n_over_tn": round(st["t2n_over_tn"], 3),
                                # a cell counts when twice the launches take at least 1.2x the time
                                "status": "ok" if st["t2n_over_tn"] >= 1.2 else "noise",
                                "pct_of_8TBs": round(100 * gbs / NOMINAL_HBM_GBS, 1),
                                "pct_of_measured_copy": round(100 * gbs / peak, 1),
                                "packed_weight_bytes": wbytes,
                                "cold": nrep * wbytes >= 2 * L2_BYTES}
                        emit(cell)
                    del reps
                    torch.cuda.empty_cache()
    # the f32 control: W ~ N(0, 0.02) drawn on the device, 4 bytes per weight
    for K in (sw["Ks"] if "f32" in parts else ()):
        for N in sw["Ns"]:
            wbytes = 4 * N * K
            todo = [M for M in sw["Ms"] if ("f32", M, N, K) not in done]
            cells += [done[("f32", M, N, K)] for M in sw["Ms"] if ("f32", M, N, K) in done]
            if not todo:
                continue
            nrep = int(min(256, max(2, -(-6 * L2_BYTES // wbytes))))
            Ws = [torch.randn((N, K), dtype=torch.float32, device="cuda", generator=gen) * 0.02 for _ in range(nrep)]
            for M in todo:
                x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=gen)
                y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                est_us = max(2.0, wbytes / 5e6)   # at about 5 TB/s
                n = int(max(nrep, min(400, 20000 / est_us)))
                st = _time_launches(torch, stream,
                                    lambda i: q4.f32gemv_run(Ws[i % nrep], x, y, M, N, K, stream=stream), n)
                byts = wbytes + 4 * M * K + 4 * M * N
                gbs = byts / st["us"] / 1e3
                emit({"kind": "f32", "M": M, "N": N, "K": K, "us_per_call": round(st["us"], 3),
                      "gbs": round(gbs, 1),
                      "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
                      "t2n_over_tn": round(st["t2n_over_tn"], 3),
                      "status": "ok" if st["t2n_over_tn"] >= 1.2 else "noise",
                      "pct_of_8TBs": round(100 * gbs / NOMINAL_HBM_GBS, 1),
                      "pct_of_measured_copy": round(100 * gbs / peak, 1),
                      "weight_bytes": wbytes, "cold": nrep * wbytes >= 2 * L2_BYTES})
            del Ws
            torch.cuda.empty_cache()
    # the read probe: prefixes of one 4 GiB buffer, 16 KiB doubling to 4 GiB
    if "probe" in parts:
        sizes = [16384 << i for i in range(19)]
        todo = [b for b in sizes if ("probe", b) not in done]
        cells += [done[("probe", b)] for b in sizes if ("probe", b) in done]
        if todo:
            pbuf = torch.rand(max(todo) // 4, dtype=torch.float32, device="cuda", generator=gen)
            partial = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
            for b in todo:
                est_us = max(2.0, b / 6e6)   # at about 6 TB/s
                n = int(max(8, min(400, 20000 / est_us)))
                st = _time_launches(torch, stream,
                                    lambda i: q4.vec4_read_probe_run(pbuf, b, partial, stream=stream), n)
                gbs = b / st["us"] / 1e3
                emit({"kind": "probe", "bytes": b, "us_per_call": round(st["us"], 3), "gbs": round(gbs, 1),
                      "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
                      "t2n_over_tn": round(st["t2n_over_tn"], 3),
                      "status": "ok" if st["t2n_over_tn"] >= 1.2 else "noise",
                      "in_l2": b <= L2_BYTES, "pct_of_measured_copy": round(100 * gbs / peak, 1)})
            del pbuf
            torch.cuda.empty_cache()
    if out is not None:
        out.close()
    big = [c for c in cells if c.get("kind", "q4") == "q4" and c["M"] == 1 and c["packed_weight_bytes"] >= 64e6]
    probe = [c for c in cells if c.get("kind") == "probe"]
    summary = {"device": device, "noise_cells": sum(1 for c in cells if c.get("status") == "noise"),"cells_m1_ge_64MB": len(big),
               "min_gbs_m1_ge_64MB": min(c["gbs"] for c in big) if big else None,
               "median_gbs_m1_ge_64MB": statistics.median(c["gbs"] for c in big) if big else None,
               "peak": peak, "peak_source": peak_src,
               "probe_max_gbs_in_l2": max((c["gbs"] for c in probe if c["in_l2"]), default=None),
               "probe_max_gbs_beyond_l2": max((c["gbs"] for c in probe if not c["in_l2"]), default=None)}
    return {"metric": "GEMV sweep (int4, f32 control) and read-probe sizes: us/call and achieved GB/s per cell",
            "unit": "GB/s",
            "launch": "overlapped" if args.overlap else "serialised", "summary": summary, "cells": cells}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.profile != "none":
        run_profile_case(args)
        return 0
    if args.sweep:
        print(json.dumps(run_sweep(args)), flush=True)
        return 0
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    res, dist = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
