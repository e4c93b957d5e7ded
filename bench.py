#!/usr/bin/env python3
"""Benchmark: int4 decode GEMV achieved HBM bandwidth on one GB300 (and N replicas).

One step = one pass of the decode projection set of a 0.5B-class transformer
at M = 1, group 32 (q, k, v, gate, up, down, LM head), each projection one
q4gemv_run call through the C ABI.  The metric is the bytes those seven GEMVs
must move (codes + scales + zero points + x + y) divided by the step time.

Timing method (after the harness lessons of cera's wgpu_gemv_bench.rs and the
Refractometer page):
  * the K timed steps are back-to-back launches on one stream, captured once in
    a CUDA graph and replayed, bracketed by CUDA events on that stream with a
    device synchronise (and a barrier across ranks) on both sides;
  * every step uses the next of several weight replicas whose total is several
    times the 129 MB L2, so each step streams its weights from HBM;
  * W untimed warm-up steps run first;
  * external event nodes inside the graph bracket the LM-head launch of every
    n-th step (--event-stride), which gives the dominant kernel's duration for
    its roofline figure; per-projection microseconds come from separate graphs
    of back-to-back launches;
  * by default the GEMVs are launched overlapped (programmatic dependent
    launch: a kernel streams its weights while the previous one finishes and
    waits for it before reading x); --overlap 0 serialises them;
  * SM clocks and throttle reasons are sampled with nvidia-smi during the
    timed region.

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

METRIC = "int4 GEMV achieved HBM GB/s (% of GB300 peak) and µs/call at M=1, 1 GPU"
UNIT = "GB/s"
WORKLOAD = "decode projection set of a 0.5B-class transformer, M=1, group=32"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu capture of
# the instance below on the LM-head shape (see profiles/); None once the kernel changes.
DOMINANT_KERNEL = "q4gemv_stream_kernel<K=896, g=32, RG=8, U=6, ASYM> (48-row blocks, 2 ring slots, 3 CTAs per SM)"
DOMINANT_TRAFFIC_BYTES = 78_731_776 + 1_214_720


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


def run_gpu(args, rank, world, local_rank):
    import torch
    import gemm_decode_gb300 as q4

    torch.cuda.set_device(local_rank)
    dist = dist_init(world, "nccl")
    q4.lib()
    q4.q4gemv_set_overlapped_launch(bool(args.overlap))
    shapes = synth.DECODE_05B["shapes"]
    group = synth.DECODE_05B["group"]
    ws = make_weights(shapes, group, synth.DECODE_05B["scale"])
    per_step_weight_bytes = sum(w.nbytes for w in ws)
    replicas = max(2, -(-args.rotate_bytes // per_step_weight_bytes))

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    reps = []
    for _ in range(replicas):
        reps.append([(to_dev(w.codes), to_dev(w.scales), to_dev(w.zeros)) for w in ws])
    xs_host = [synth.activations_f32(77 + i, 1, K) for i, (_, _, K) in enumerate(shapes)]
    xs = [to_dev(x) for x in xs_host]
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in shapes]

    stream = torch.cuda.Stream()
    ev = GraphEvents(torch)

    LM = len(shapes) - 1   # the dominant launch: the LM head

    def one_step(r, s, events=None, i_step=0, only=None):
        for p, ((name, N, K), w) in enumerate(zip(shapes, ws)):
            c, sc, z = reps[r][p]
            timed = events is not None and (only is None or p == only)
            if timed:
                ev.record(events[i_step][p][0], s)
            q4.q4gemv_run(c, sc, z, xs[p], ys[p], 1, N, K, group, stream=s)
            if timed:
                ev.record(events[i_step][p][1], s)

    # eager pass (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for r in range(replicas):
            one_step(r, stream)
    torch.cuda.synchronize()

    chunk = min(args.steps, max(replicas, args.graph_steps))
    chunk = max(1, chunk)
    reps_timed = args.steps // chunk
    tail = args.steps - reps_timed * chunk
    events = [[(ev.new(), ev.new()) for _ in shapes] for _ in range(chunk)]
    # LM-head launches bracketed by event nodes: every stride-th step of the timed graph
    # (an event node costs a bubble and breaks the launch overlap around it)
    stride = max(1, min(args.event_stride, chunk))
    sampled = list(range(0, chunk, stride))

    def capture(n, with_events, offset=0, only=LM):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                timed = with_events and i % stride == 0
                one_step((offset + i) % replicas, stream, events if timed else None, i, only)
        return g

    g_main = capture(chunk, True)
    g_tail = capture(tail, False, offset=chunk * reps_timed) if tail else None

    # warm-up: exactly W steps (a graph of min(W, chunk) steps, replayed, plus a remainder)
    if args.warmup:
        wn = min(args.warmup, chunk)
        g_warm = capture(wn, False)
        wfull, wtail = divmod(args.warmup, wn)
        g_wtail = capture(wtail, False) if wtail else None
        with torch.cuda.stream(stream):
            for _ in range(wfull):
                g_warm.replay()
            if g_wtail is not None:
                g_wtail.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(smi_index(local_rank)).start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps_timed):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier(dist)
    clocks = sampler.stop(t0, t1)
    ms_total = start.elapsed_time(end)
    ms_total_max = reduce_over_ranks(dist, ms_total, "max", device="cuda")

    # the dominant launch's duration: event nodes around each LM-head launch of the
    # last replay of the timed graph (the only event nodes in it)
    lm_us = statistics.fmean(ev.elapsed_ms(events[i][LM][0], events[i][LM][1]) * 1e3 for i in sampled)
    # per-projection microseconds per call: for each projection, one graph of back-to-back
    # launches over the rotating replicas, timed from outside (no event nodes between
    # launches; event nodes cost a bubble of about a microsecond or more each)
    per_proj = []
    n_pp = max(replicas, min(args.steps, 200))
    for p, (name, N, K) in enumerate(shapes):
        per_proj.append(_time_back_to_back(torch, q4, stream, [r[p] for r in reps], xs[p], ys[p], 1, N, K, group,
                                           n_pp))
    bytes_per_step = step_bytes(shapes, 1, group)
    total_bytes = bytes_per_step * args.steps * world
    value = total_bytes / (ms_total_max * 1e-3) / 1e9
    ms_per_step = ms_total_max / args.steps

    peak, peak_src = load_peaks()
    lm_bytes = algorithmic_bytes(1, shapes[LM][1], shapes[LM][2], group)
    # the dominant kernel's launch duration: CUDA events on its launching stream around
    # a graph of back-to-back LM-head launches (rotating replicas, cold L2, overlapped
    # launch as in the step), timed in this run right after the timed region.  The
    # in-step figure (event nodes around sampled LM-head launches of the timed graph)
    # is reported beside it: those nodes break the launch overlap and add a bubble.
    lm_b2b_us = per_proj[LM]["us"]
    achieved = lm_bytes / (lm_b2b_us * 1e-6) / 1e9
    in_step = lm_bytes / (lm_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": DOMINANT_KERNEL + " on lm_head 151936x896",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": args.traffic_bytes if args.traffic_bytes is not None else DOMINANT_TRAFFIC_BYTES,
                "algorithmic_bytes_per_launch": lm_bytes,
                "duration_us": round(lm_b2b_us, 3),
                "duration_source": "CUDA events on the launching stream around a graph of back-to-back "
                                   "LM-head launches (rotating replicas, cold L2, overlapped launch), "
                                   "median of 5 replays, right after the timed region",
                "in_step": {"us": round(lm_us, 3), "achieved": round(in_step, 1),
                            "frac": round(in_step / peak, 4),
                            "how": "event nodes around the LM-head launch of every "
                                   f"{stride}th timed step; they break the launch overlap "
                                   "and add a bubble, so this figure is conservative"}}

    # ---- end to end: pinned host x in, pinned host y out, through the same API ----
    e2e = run_e2e(args, torch, q4, shapes, group, reps, xs_host, replicas, stream, dist)

    detail = {"projections": [
        {"name": name, "N": N, "K": K, "us_per_call": round(st["us"], 3),
         "gbs": round(algorithmic_bytes(1, N, K, group) / (st["us"] * 1e-6) / 1e9, 1),
         "us_p10_p90_min": [round(st["p10"], 3), round(st["p90"], 3), round(st["min"], 3)],
         "t2n_over_tn": round(st["t2n_over_tn"], 3)}
        for (name, N, K), st in zip(shapes, per_proj)],
        "weight_replicas": replicas, "replica_bytes": per_step_weight_bytes,
        "graph_steps": chunk, "event_mode": ev.mode,
        "lm_head_us_in_timed_region": round(lm_us, 3),
        "lm_head_event_samples": f"{len(sampled)} per {chunk}-step graph (every {stride}th step)",
        "us_per_call_note": "per projection: a graph of back-to-back launches over the rotating replicas, "
                            "5 timed replays (median; p10, p90, min) and t(2n)/t(n) from two replays; "
                            "the LM head's in-step time carries the event-node bubble"}
    if args.controls and rank == 0:
        detail["controls"] = run_controls(args, torch, q4)
        detail["prefill_tensor_core"] = run_prefill(args, torch, q4)
        detail["decode_8b"] = run_decode_8b(args, torch, q4)
        detail["fused_projections_step"] = run_fused_step(args, torch, q4, shapes, group, reps, xs, replicas,
                                                          stream)
        detail["q4_0_format"] = run_q40(args, torch, q4)
        try:   # a detail figure: its failure is recorded, the measured step stands
            detail["grouped_step"] = run_grouped_step(args, torch, q4, shapes, group, reps, xs, replicas, stream)
        except Exception as e:   # noqa: BLE001
            detail["grouped_step"] = {"error": f"{type(e).__name__}: {e}"}

    probe = detail.get("controls", {}).get("vec4_read_probe_1GiB", {}).get("gbs")
    if probe:   # the same kernel's rate against this GPU's own streaming read (the vec4 probe)
        roofline["frac_of_read_probe"] = round(roofline["achieved"] / probe, 4)
        roofline["read_probe_gbs"] = probe
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights (fp16 scales, u4 zeros), f32 x/accumulate/y",
        "data": "synthetic (seeded; codes/zeros uniform 0..15, scales fp16 U[0.005,0.02], x N(0,1))",
        "config": {"workload": WORKLOAD, "M": 1, "group": group,
                   "shapes": [[n, N, K] for n, N, K in shapes],
                   "bytes_per_step": bytes_per_step,
                   "l2_policy": f"inputs larger than L2: {replicas} rotating weight replicas "
                                f"({replicas * per_step_weight_bytes / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": ("overlapped: programmatic dependent launch, each GEMV waits for the "
                              "previous kernel before reading x" if args.overlap else "serialised")},
        "clocks": clocks, "e2e": e2e, "gpu_launches": len(shapes) * args.steps,
        "roofline": roofline, "pct_of_8TBs_nominal": round(value / NOMINAL_HBM_GBS, 4),
        "detail": detail,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, ws, xs_host, shapes, group,
                                              gpu_outputs=[y.cpu().numpy() for y in ys])
    return result, dist


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
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(full):
                g.replay()
            if gt is not None:
                gt.replay()
            end.record(stream)
        torch.cuda.synchronize()
        return reduce_over_ranks(dist, start.elapsed_time(end), "max", device="cuda")

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

    hows = {"copy": "CUDA graph of K steps: pinned-host x -> device copy, 7 x q4gemv_run, y -> pinned host copy",
            "mapped": "CUDA graph of K steps; 7 x q4gemv_run reading x from and writing y to pinned host memory "
                      "(NVLink-C2C, no copy nodes)",
            "x_copy_y_mapped": "CUDA graph of K steps: pinned-host x -> device copy, 7 x q4gemv_run writing y "
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
    measured dense bf16 peak (2*M*N*K flops per call)."""
    out = []
    burst, sustained, src = load_bf16_peak()
    for name, M, N, K in synth.PREFILL["shapes"]:
        w = synth.q4_weights(7, N, K, 32, tag=name)
        a = synth.activations_bf16(7, M, K)
        dev = lambda x: None if x is None else torch.from_numpy(
            np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
        cw, sw, zw, ad = dev(w.codes), dev(w.scales), dev(w.zeros), dev(a)
        c = torch.empty((M, N), dtype=torch.float32, device="cuda")
        n_it = 20 if M * N * K > 1e10 else 200
        for _ in range(3):
            q4.q4gemm_run(cw, sw, zw, ad, c, M, N, K, 32)
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(n_it):
            q4.q4gemm_run(cw, sw, zw, ad, c, M, N, K, 32)
        e0.record()
        torch.cuda.synchronize()
        assert q4.q4gemv_device_status() == q4.Q4_OK
        us = s0.elapsed_time(e0) * 1e3 / n_it
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out.append({"name": name, "M": M, "N": N, "K": K, "us": round(us, 2), "tflops": round(tf, 1),
                    "frac_of_bf16_peak": round(tf / burst, 4), "peak": burst, "peak_source": src,
                    "note": "back-to-back calls on one weight copy (W fits in L2)"})
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
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    outs, nbytes = oracle_step(ws, xs_host, shapes, group, threads)
    dt = time.perf_counter() - t0
    steps = 1
    while time.perf_counter() - t0 < args.cpu_seconds:
        oracle_step(ws, xs_host, shapes, group, threads)
        steps += 1
    dt = time.perf_counter() - t0
    res = {"value": round(nbytes * steps / dt / 1e9, 4), "unit": UNIT, "cores": threads,
           "kind": "oracle",
           "sample": f"{steps} full step(s) of the projection set (all rows), "
                     f"{threads} threads over row slices, {dt:.1f} s wall"}
    if gpu_outputs is not None:
        worst = 0.0
        for (y_ref, bound), y in zip(outs, gpu_outputs):
            err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
            worst = max(worst, float(np.max(err / (1e-3 * bound + 1e-6))))
        res["parity_gate"] = {"max_err_over_bound": round(worst, 6), "ok": worst <= 1.0}
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
    shapes = synth.DECODE_05B["shapes"]
    group = synth.DECODE_05B["group"]
    ws = make_weights(shapes, group, synth.DECODE_05B["scale"])
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
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
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
                                         "tc_lm05_m8", "tc_down8b_m8", "f32_lm_head", "gemm_ffn", "gemm_gate"],
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
    "tc_m16": (32768, 4096, 128, 16),      # tensor-core GEMV, 128-row tiles, no K split
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

    n = max(replicas, min(args.steps, 2000))
    with torch.cuda.stream(stream):
        for r in range(replicas):
            step(r)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            step(i % replicas)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    byts = step_bytes(fshapes, 1, group)
    out = {"launches_per_step": len(fshapes), "shapes": [[nm, N, K] for nm, N, K in fshapes],
           "us_per_step": round(us, 3), "gbs": round(byts / us / 1e3, 1), "bytes_per_step": byts}

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

    with torch.cuda.stream(stream):
        for r in range(replicas):
            step_fused(r)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for i in range(n):
            step_fused(i % replicas)
    with torch.cuda.stream(stream):
        g2.replay()
        e0.record(stream)
        g2.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us2 = e0.elapsed_time(e1) * 1e3 / n
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
    """The same seven projections, each with its own x and y as in the timed step, issued
    through q4gemv_grouped_run: the six K = 896 matrices (q, k, v, gate, up, LM head) as
    one streamed launch in which each has CTAs of its own, down (K = 4864) as a second.
    A CUDA graph of back-to-back steps over the replicas; the outputs are checked against
    the separate calls' within the GEMV tolerance by the tests, not here."""
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in shapes]
    byK = {}
    for p, (_, N, K) in enumerate(shapes):
        byK.setdefault(K, []).append(p)

    def step(r):
        for K, ps in byK.items():
            q4.q4gemv_grouped_run([(*reps[r][p], xs[p], ys[p], shapes[p][1]) for p in ps], K, group, stream=stream)

    n = max(replicas, min(args.steps, 2000))
    with torch.cuda.stream(stream):
        for r in range(replicas):
            step(r)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            step(i % replicas)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    byts = step_bytes(shapes, 1, group)
    return {"calls_per_step": len(byK), "groups": {str(K): [shapes[p][0] for p in ps] for K, ps in byK.items()},
            "us_per_step": round(us, 3), "gbs": round(byts / us / 1e3, 1), "bytes_per_step": byts}


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
