#!/usr/bin/env python3
"""Benchmark of the weight-only quantized linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--headline-only] [--no-cpu-baseline]
                    [--only nvfp4|gemm|grouped|w8a8|gemv-shapes]

Prints ONE JSON line (rank 0).  The headline `value` is the M=1 FP8 (W8A16)
decode GEMV throughput in GB/s of algorithmic bytes over one step = the three
decode shapes (N, K) = (4096, 4096), (14336, 4096), (4096, 14336), bf16 output
with the per-tensor scale folded.  The same line carries, under "sub", the
other halves of the metric (NVFP4 GEMV GB/s, M=2048 W8A16 GEMM TFLOP/s), the
NVFP4 M=16/128 GEMMs, the FP8 GEMM with K = 4100, the FP8 and NVFP4
grouped-MoE GEMMs and the W8A8 int8 quantizer + GEMM, each with its
roofline fraction against MEASURED_PEAKS.json.

Timing: inputs are resident in HBM; the K timed steps run as CUDA-graph
replays (a captured chunk of steps, replayed until exactly K steps ran),
bracketed by a barrier and torch.cuda.synchronize() on both sides, timed with
CUDA events on the launching stream, max over ranks.  L2 (129 MB) is defeated
by rotating several device copies of the weights so that one rotation is well
above the L2 size; each step reads a copy that was evicted since it was last
read.  SM clocks and throttle reasons are sampled with nvidia-smi during the
timed region.

`--impl reference` times the CPU oracle (the plain float64 definition in
oracle/) on the host cores on the same workload and metric: a bounded sample
of each step (stated in the line), the only other place this script runs it.

Multi-GPU: the layer does not shard in this build ("replicas only"): with
--gpus N each rank runs the same per-GPU work on its own GPU and the value is
the sum of the ranks' bytes over the slowest rank's time (scaling "weak").
"""

from __future__ import annotations

import argparse
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
import torch  # noqa: E402

METRIC = "M=1 FP8/NVFP4 GEMV HBM GB/s (% of peak); M=2048 W8A16 GEMM TFLOP/s"
GEMV_SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336)]
L2_BYTES = 129 * 1024 * 1024
ROTATION_TARGET = 4 * L2_BYTES          # bytes of weights in one rotation


# ------------------------------------------------------------ distributed --

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def aggregate(world, units: float, ms: float, device="cpu"):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    if world == 1:
        return units, ms
    t = torch.tensor([units, ms], dtype=torch.float64, device=device)
    u = t[0:1].clone()
    m = t[1:2].clone()
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    torch.distributed.all_reduce(m, op=torch.distributed.ReduceOp.MAX)
    return float(u.item()), float(m.item())


# ----------------------------------------------------------------- peaks --

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_index: int, period_ms: int = 20):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        self.gpu = ids[local_index] if local_index < len(ids) else str(local_index)
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let nvidia-smi attach before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ timing --

# Set by our arm to gq.device_status: every timed region is followed by a read
# of the library's status word, and a run in which any bounded in-kernel wait
# gave up (the kernel then returns early with partial results) is an error,
# never a figure.
STATUS_CHECK = None


def check_device_status(what: str):
    if STATUS_CHECK is None:
        return
    st = STATUS_CHECK()
    if st != 0:
        raise RuntimeError(f"{what}: a kernel wait timed out (device status {st:#x}); "
                           "the timing is invalid")


def graph_timer(step_fn, steps, warmup, chunk, stream, world, sampler=None):
    """Run `warmup` eager steps, capture `chunk` steps into a CUDA graph and
    replay until exactly `steps` ran (the remainder as a second, shorter
    graph).  Returns the elapsed ms of the K timed steps (CUDA events on
    `stream`); raises if a kernel reported a timed-out wait meanwhile."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            step_fn(i)
    torch.cuda.synchronize()
    chunk = max(1, min(chunk, steps))
    graphs = []
    full, rem = divmod(steps, chunk)
    for n in ([chunk] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step_fn(i)
        with torch.cuda.stream(stream):
            g.replay()                  # untimed: uploads the graph
        graphs.append((g, n))
    torch.cuda.synchronize()
    order = [graphs[0][0]] * full if full else []
    if rem:
        order.append(graphs[-1][0])
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):         # replay on the stream the events time
        start.record(stream)
        for g in order:
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.stop()
    check_device_status("timed region")
    return start.elapsed_time(end)


# --------------------------------------------------------------- workloads --

def n_copies(bytes_per_set: int) -> int:
    return max(2, int(math.ceil(ROTATION_TARGET / max(1, bytes_per_set))))


def copies_past_l2(bytes_per_copy: int) -> int:
    """Rotating copies of a sub-benchmark's inputs so that one rotation reads
    at least twice the L2 capacity (consecutive launches find nothing of
    their inputs in L2)."""
    return max(2, int(math.ceil(2 * L2_BYTES / max(1, bytes_per_copy))))


def make_fp8_gemv_sets(dev):
    import synth
    base = []
    for i, (n, k) in enumerate(GEMV_SHAPES):
        codes, s = synth.fp8_weight(n, k, seed=0)
        x = synth.bf16_activations(1, k, seed=1).reshape(-1)
        base.append((codes, s, x))
    set_bytes = sum(n * k for n, k in GEMV_SHAPES)
    copies = n_copies(set_bytes)
    sets = []
    for c in range(copies):
        sets.append([(codes.to(dev), s, x.to(dev)) for codes, s, x in base])
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for n, _ in GEMV_SHAPES]
    return base, sets, outs, copies


def fp8_gemv_bytes(n, k):
    return n * k + 2 * k + 2 * n          # weights + bf16 x + bf16 y


def nvfp4_bytes(m, n, k):
    return n * k // 2 + n * k // 16 + 2 * m * k + 2 * m * n


# -------------------------------------------------------------- our arm --

def run_ours(args, rank, local, world):
    import gemm_fp8_nvfp4_gb300 as gq
    global STATUS_CHECK
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    gq.load_library()
    STATUS_CHECK = gq.device_status
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    launches = {"n": 0}

    # ---------------- headline: FP8 decode GEMV over the three shapes
    base, sets, outs, copies = make_fp8_gemv_sets(dev)
    step_bytes = sum(fp8_gemv_bytes(n, k) for n, k in GEMV_SHAPES)

    def gemv_step(i):
        st = sets[i % copies]
        for j, (w, s, x) in enumerate(st):
            gq.fp8_gemv(x, w, s, out=outs[j], stream=stream)

    sampler = ClockSampler(local)
    if args.overlap_weight_reads:
        gq.set_launch_flags(gq.GQ_LAUNCH_OVERLAP_WEIGHT_READS)
    ms = graph_timer(gemv_step, args.steps, args.warmup, min(200, args.steps), stream, world,
                     sampler)
    gemv_launches = 3 * args.steps
    total_bytes, ms_max = aggregate(world, step_bytes * args.steps, ms, device=dev)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    clocks = sampler.summary()

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "operands": {"weights": "float8_e4m3fn", "activations": "bf16", "out": "bf16",
                     "accumulate": "f32"},
        "data": "synthetic (seeded: W ~ N(0,0.02) quantized per tensor to e4m3, x ~ N(0,1) bf16)",
        "config": {
            "workload": "FP8 W8A16 decode GEMV, M=1, (N,K) in {(4096,4096),(14336,4096),"
                        "(4096,14336)}, bf16 out, per-tensor scale folded",
            "step": "one GEMV per shape (3 launches)",
            "l2": f"inputs larger than L2: {copies} rotating weight copies "
                  f"({copies * sum(n * k for n, k in GEMV_SHAPES) / 1e6:.0f} MB per rotation)",
            "timing": "CUDA-graph replay, CUDA events on the launching stream",
            "launch": ("GQ_LAUNCH_OVERLAP_WEIGHT_READS (weight reads overlap the previous GEMV)"
                       if args.overlap_weight_reads else "plain stream order"),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(value / world, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(value / world / peaks["hbm_gbs"], 4),
            "peak_source": peaks["source"],
            "kernel": "k_fp8_gemv<16,R,U,128> (R x U = 8 x 2 for K = 4096, 4 x 4 for K = 14336)",
            "traffic": committed_traffic("fp8_gemv"),
            "frac_of_nominal_8tbs": round(value / world / 8000.0, 4),
        },
        "gpu_launches": gemv_launches,
        "clocks": clocks,
    }

    # The HBM floor of the same launches: each GEMV's kernel in its launch
    # shape with the weight loads only (gq_probe_gemv_read_floor), same
    # rotation, same replay.
    def floor_step(i):
        st = sets[i % copies]
        for j, (w, s, x) in enumerate(st):
            gq.probe_gemv_read_floor(w, out=outs[j], stream=stream)

    ms_f = graph_timer(floor_step, args.steps, args.warmup, min(200, args.steps), stream, world)
    _, ms_f = aggregate(world, step_bytes * args.steps, ms_f, device=dev)
    line["roofline"]["floor"] = {
        "what": "the same three launches with the loads only (gq_probe_gemv_read_floor)",
        "ms_per_step": ms_f / args.steps,
        "GB/s": round(step_bytes * args.steps / (ms_f * 1e-3) / 1e9, 1),
        "frac": round(step_bytes * args.steps / (ms_f * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "value_over_floor": round(ms_f / ms_max, 4)}

    if not args.overlap_weight_reads and not args.headline_only:
        # The same step with GQ_LAUNCH_OVERLAP_WEIGHT_READS (decode with fixed
        # weights: each GEMV's weight reads overlap the previous kernel).
        gq.set_launch_flags(gq.GQ_LAUNCH_OVERLAP_WEIGHT_READS)
        ms_o = graph_timer(gemv_step, args.steps, args.warmup, min(200, args.steps), stream, world)
        gq.set_launch_flags(0)
        tb_o, ms_o = aggregate(world, step_bytes * args.steps, ms_o, device=dev)
        v_o = tb_o / (ms_o * 1e-3) / 1e9
        line["overlap_weight_reads"] = {
            "value": round(v_o, 1), "unit": "GB/s", "ms_per_step": ms_o / args.steps,
            "frac": round(v_o / world / peaks["hbm_gbs"], 4),
            "note": "same step with GQ_LAUNCH_OVERLAP_WEIGHT_READS: valid when no kernel "
                    "between GEMVs writes their weights (decode with fixed weights)"}
    if not args.headline_only:
        line["sub"] = run_subs(args, gq, dev, stream, peaks, world)
        line["gpu_launches"] = gemv_launches  # the timed region of the headline only

    # ---------------- end to end: host buffers, copies inside the timed region
    line["e2e"] = e2e_gemv(gq, base, dev, stream, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_gemv(args)
        if not args.headline_only:
            line["cpu_baseline"]["per_config"] = cpu_baseline_configs()
    line["device_status"] = gq.device_status()   # 0: no in-kernel wait gave up
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def committed_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel source is unchanged since the capture (hash recorded beside it)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if not ent:
            return None
        import hashlib
        src = os.path.join(ROOT, ent["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return ent["bytes_per_launch"] if h == ent["source_sha256_16"] else None
    except Exception:
        return None


def e2e_gemv(gq, base, dev, stream, args, world):
    """The headline metric through the public API from pinned host buffers:
    every step copies the step's weights and activations host -> device,
    runs the three GEMVs and copies the outputs back.  The host -> device
    copies run on a copy stream into two device buffer sets used by
    alternate steps, so the copies of step i + 1 overlap the GEMVs and the
    device -> host copies of step i; each GEMV waits only for its own
    operands, and a buffer set is refilled only after the GEMVs that read
    it two steps earlier have finished."""
    host = [(codes.pin_memory(), s, x.pin_memory()) for codes, s, x in base]
    nbuf = 2
    dbufs = [[(torch.empty_like(c, device=dev), torch.empty_like(x, device=dev))
              for c, _, x in host] for _ in range(nbuf)]
    outs_h = [[torch.empty(n, dtype=torch.bfloat16).pin_memory() for n, _ in GEMV_SHAPES]
              for _ in range(nbuf)]
    outs_d = [[torch.empty(n, dtype=torch.bfloat16, device=dev) for n, _ in GEMV_SHAPES]
              for _ in range(nbuf)]
    h2d = sum(c.numel() + 2 * x.numel() for c, _, x in host)
    d2h = sum(2 * n for n, _ in GEMV_SHAPES)
    steps = max(3, min(args.steps, 50))
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [[torch.cuda.Event() for _ in host] for _ in range(nbuf)]
    done = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def step(i):
        b = i % nbuf
        with torch.cuda.stream(copy_stream):
            if used[b]:
                copy_stream.wait_event(done[b])
            for j, (c, _, x) in enumerate(host):
                dbufs[b][j][0].copy_(c, non_blocking=True)
                dbufs[b][j][1].copy_(x, non_blocking=True)
                ready[b][j].record(copy_stream)
        with torch.cuda.stream(stream):
            for j, (_, s, _) in enumerate(host):
                stream.wait_event(ready[b][j])
                gq.fp8_gemv(dbufs[b][j][1], dbufs[b][j][0], s, out=outs_d[b][j], stream=stream)
                outs_h[b][j].copy_(outs_d[b][j], non_blocking=True)
            done[b].record(stream)
        used[b] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for i in range(steps):
        step(i)
    e1.record(stream)   # after the last step's GEMVs, which follow every copy
    torch.cuda.synchronize()
    barrier(world)
    check_device_status("end-to-end run")
    ms = e0.elapsed_time(e1)
    step_bytes = sum(fp8_gemv_bytes(n, k) for n, k in GEMV_SHAPES)
    total, ms_max = aggregate(world, step_bytes * steps, ms, device=dev)
    return {"value": round(total / (ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "note": ("pinned host buffers; per step the H2D of weights + x, 3 GEMVs and the D2H "
                     "of y; H2D on a copy stream, double-buffered across steps")}


def run_subs(args, gq, dev, stream, peaks, world, only=None):
    import synth
    subs = {}
    steps = max(20, min(args.steps, 200)) if only is None else args.steps
    warm = max(3, min(args.warmup, 10))
    gsteps = max(10, min(args.steps, 50)) if only is None else args.steps

    # NVFP4 GEMV / small-M GEMM, N = K = 4096, M in {1, 16, 128}
    if only in (None, "nvfp4"):
        nvfp4_subs(gq, dev, stream, peaks, world, steps, warm, subs)
    if only in (None, "gemm"):
        gemm_sub(gq, dev, stream, peaks, world, gsteps, warm, subs)
    if only in (None, "grouped"):
        grouped_sub(gq, dev, stream, peaks, world, gsteps, warm, subs)
    if only in (None, "w8a8"):
        w8a8_sub(gq, dev, stream, peaks, world, gsteps, warm, subs)
    return subs


def nvfp4_subs(gq, dev, stream, peaks, world, steps, warm, subs):
    import synth
    n = k = 4096
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=0)
    copies = n_copies(n * k // 2 + n * k // 16)
    qs = [(q.to(dev), bs.to(dev)) for _ in range(copies)]
    for m in (1, 16, 128):
        a = synth.bf16_activations(m, k, seed=1).to(dev)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        if m == 1:
            def step(i, a=a, out=out):
                qq, bb = qs[i % copies]
                gq.nvfp4_gemv(a.reshape(-1), qq, bb, s2, out=out.reshape(-1), stream=stream)
        else:
            def step(i, a=a, out=out):
                qq, bb = qs[i % copies]
                gq.nvfp4_matmul(a, qq, bb, s2, out=out, stream=stream)
        ms = graph_timer(step, steps, warm, steps, stream, world)
        t = ms * 1e-3 / steps
        gbs = nvfp4_bytes(m, n, k) / t / 1e9
        floor = None
        if m == 1:
            def fstep(i, out=out):
                qq, bb = qs[i % copies]
                gq.probe_gemv_read_floor(qq, bb, out=out.reshape(-1), stream=stream)
            tf = graph_timer(fstep, steps, warm, steps, stream, world) * 1e-3 / steps
            floor = {"what": "the same launch with the loads only (gq_probe_gemv_read_floor)",
                     "us": round(tf * 1e6, 3), "frac_hbm": round(nvfp4_bytes(m, n, k) / tf / 1e9 /
                                                                   peaks["hbm_gbs"], 4),
                     "time_over_floor": round(t / tf, 4)}
        tfl = 2 * m * n * k / t / 1e12
        key = "nvfp4_gemv_m1" if m == 1 else f"nvfp4_gemm_m{m}"
        frac_hbm = gbs / peaks["hbm_gbs"]
        frac_tc = tfl / peaks["bf16_tflops"]
        subs[key] = {"us_per_launch": round(t * 1e6, 3), "GB/s": round(gbs, 1),
                     "TFLOP/s": round(tfl, 2), "frac_hbm": round(frac_hbm, 4),
                     "frac_bf16_tensor": round(frac_tc, 4),
                     "roofline_frac": round(max(frac_hbm, frac_tc) if m == 128 else frac_hbm, 4),
                     "l2": f"{copies} rotating weight copies"}
        if floor is not None:
            subs[key]["floor"] = floor
            subs[key]["traffic"] = committed_traffic("nvfp4_gemv")
    del qs


def gemm_sub(gq, dev, stream, peaks, world, gsteps, warm, subs):
    """FP8 GEMM M=2048 N=14336 K=4096."""
    import synth
    m, n, k = 2048, 14336, 4096
    codes, s = synth.fp8_weight(n, k, seed=0)
    a = synth.bf16_activations(m, k, seed=1)
    copies = copies_past_l2(n * k + 2 * m * k)
    ins = [(a.to(dev), codes.to(dev)) for _ in range(copies)]
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

    def gemm_step(i):
        aa, ww = ins[i % copies]
        gq.fp8_matmul(aa, ww, s, out=out, stream=stream)

    ms = graph_timer(gemm_step, gsteps, warm, gsteps, stream, world)
    t = ms * 1e-3 / gsteps
    tfl = 2 * m * n * k / t / 1e12
    subs["fp8_gemm_m2048"] = {"us_per_launch": round(t * 1e6, 2), "TFLOP/s": round(tfl, 1),
                              "frac_bf16_tensor": round(tfl / peaks["bf16_tflops"], 4),
                              "frac_bf16_tensor_sustained":
                                  round(tfl / peaks["bf16_tflops_sustained"], 4),
                              "l2": f"{copies} rotating input copies"}
    del ins

    # The same product with K = 4100 and 4104 (rows not 16-byte strided):
    # the residue-class staging path (4104: A by the plain tiled box).
    for k2 in (4100, 4104):
        codes2, s2 = synth.fp8_weight(n, k2, seed=0)
        a2 = synth.bf16_activations(m, k2, seed=1)
        ins2 = [(a2.to(dev), codes2.to(dev)) for _ in range(copies)]

        def anyk_step(i, ins2=ins2, s2=s2):
            aa, ww = ins2[i % copies]
            gq.fp8_matmul(aa, ww, s2, out=out, stream=stream)

        ms = graph_timer(anyk_step, gsteps, warm, gsteps, stream, world)
        t = ms * 1e-3 / gsteps
        tfl = 2 * m * n * k2 / t / 1e12
        subs[f"fp8_gemm_m2048_k{k2}"] = {"us_per_launch": round(t * 1e6, 2),
                                         "TFLOP/s": round(tfl, 1),
                                         "frac_bf16_tensor": round(tfl / peaks["bf16_tflops"], 4),
                                         "l2": f"{copies} rotating input copies"}
        del ins2


def w8a8_sub(gq, dev, stream, peaks, world, gsteps, warm, subs):
    """W8A8 int8 (the sibling method): per-row activation quantization of
    x [2048, 4096] bf16, then the int8 GEMM with W [14336, 4096] int8."""
    import synth
    m, n, k = 2048, 14336, 4096
    qb, sb = synth.int8_weight(n, k, seed=0)
    x = synth.bf16_activations(m, k, seed=1)
    copies = copies_past_l2(n * k + 2 * m * k)
    ins = [(x.to(dev), qb.to(dev)) for _ in range(copies)]
    # The quantizer reads only x: enough copies of it alone to exceed L2.
    xcopies = copies_past_l2(2 * m * k)
    xs = [x.to(dev) for _ in range(xcopies)]
    d_sb = sb.to(dev)
    qa = torch.empty((m, k), dtype=torch.int8, device=dev)
    sa = torch.empty((m,), dtype=torch.float32, device=dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

    def quant_step(i):
        gq.int8_quantize_rows(xs[i % xcopies], q=qa, scale=sa, stream=stream)

    def gemm_step(i):
        gq.int8_matmul(qa, ins[i % copies][1], sa, d_sb, out=out, stream=stream)

    def both_step(i):
        quant_step(i)
        gemm_step(i)

    tq = graph_timer(quant_step, gsteps, warm, gsteps, stream, world) * 1e-3 / gsteps
    tg = graph_timer(gemm_step, gsteps, warm, gsteps, stream, world) * 1e-3 / gsteps
    tb = graph_timer(both_step, gsteps, warm, gsteps, stream, world) * 1e-3 / gsteps
    qbytes = 2 * m * k + m * k + 4 * m
    tfl = 2 * m * n * k / tg / 1e12
    subs["int8_w8a8_m2048"] = {
        "quantize_us": round(tq * 1e6, 2),
        "quantize_GB/s": round(qbytes / tq / 1e9, 1),
        "quantize_frac_hbm": round(qbytes / tq / 1e9 / peaks["hbm_gbs"], 4),
        "gemm_us": round(tg * 1e6, 2), "gemm_TFLOP/s": round(tfl, 1),
        "gemm_frac_bf16_tensor": round(tfl / peaks["bf16_tflops"], 4),
        "step_us": round(tb * 1e6, 2),
        "l2": f"{xcopies} rotating activation copies (quantizer), {copies} rotating input copies (GEMM)"}
    del ins, xs


def grouped_sub(gq, dev, stream, peaks, world, gsteps, warm, subs):
    """Grouped MoE, FP8 then NVFP4: 8 experts [8, 14336, 4096], 4096 routed rows."""
    import synth
    stack, scales = synth.fp8_expert_stack(8, 14336, 4096, seed=0)
    a = synth.bf16_activations(4096, 4096, seed=1)
    offs, ids, counts = synth.moe_routing(4096, seed=2)
    d_stack, d_scales, d_a = stack.to(dev), scales.to(dev), a.to(dev)
    d_offs = offs.to(torch.int32).to(dev)
    d_ids = ids.to(torch.int32).to(dev)
    outg = torch.empty((4096, 14336), dtype=torch.bfloat16, device=dev)
    active_rows = int(counts[:-1].sum())

    def grouped_step(i):
        gq.fp8_grouped_matmul(d_a, d_stack, d_offs, d_ids, d_scales,
                              max_rows_per_group=int(counts.max()), out=outg, stream=stream)

    ms = graph_timer(grouped_step, gsteps, warm, gsteps, stream, world)
    t = ms * 1e-3 / gsteps
    tfl = 2 * 14336 * 4096 * active_rows / t / 1e12
    subs["fp8_grouped_moe"] = {"us_per_launch": round(t * 1e6, 2), "TFLOP/s": round(tfl, 1),
                               "frac_bf16_tensor": round(tfl / peaks["bf16_tflops"], 4),
                               "active_rows": active_rows,
                               "l2": "weights 470 MB > L2"}
    del d_stack

    # The same routing with NVFP4 experts (q [8, 14336, 2048], bs [8, 14336, 256]).
    q, bs, s2 = synth.nvfp4_expert_stack(8, 14336, 4096, seed=0)
    d_q, d_bs, d_s2 = q.to(dev), bs.to(dev), s2.to(dev)

    def nvfp4_grouped_step(i):
        gq.nvfp4_grouped_matmul(d_a, d_q, d_bs, d_offs, d_ids, d_s2,
                                max_rows_per_group=int(counts.max()), out=outg, stream=stream)

    ms = graph_timer(nvfp4_grouped_step, gsteps, warm, gsteps, stream, world)
    t = ms * 1e-3 / gsteps
    tfl = 2 * 14336 * 4096 * active_rows / t / 1e12
    subs["nvfp4_grouped_moe"] = {"us_per_launch": round(t * 1e6, 2), "TFLOP/s": round(tfl, 1),
                                 "frac_bf16_tensor": round(tfl / peaks["bf16_tflops"], 4),
                                 "active_rows": active_rows,
                                 "l2": "weights 264 MB > L2"}


# -------------------------------------------------------------- CPU oracle --

def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_gemv(args, budget_s=12.0):
    """The oracle as it stands, timed on this host's cores on the headline
    workload: whole steps (the three decode shapes) until ~budget_s."""
    import oracle
    import synth
    inputs = []
    for n, k in GEMV_SHAPES:
        codes, s = synth.fp8_weight(n, k, seed=0)
        x = synth.bf16_activations(1, k, seed=1).reshape(-1)
        inputs.append((codes.numpy(), s, synth.bf16_bits(x)))
    step_bytes = sum(fp8_gemv_bytes(n, k) for n, k in GEMV_SHAPES)
    t0 = time.perf_counter()
    steps = 0
    while True:
        for codes, s, xb in inputs:
            oracle.fp8_gemv(xb, codes, s)
        steps += 1
        if time.perf_counter() - t0 > budget_s or steps >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": round(step_bytes * steps / dt / 1e9, 3), "unit": "GB/s",
            "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{steps} full step(s) of the three decode shapes in {dt:.1f} s "
                      f"(numpy float64 table decode + matvec)"}


def cpu_baseline_configs():
    """The oracle timed on the other workloads of the line (each a bounded,
    stated sample), in the unit of the matching sub-result."""
    import oracle
    import synth

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    out = {}
    n = k = 4096
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=0)
    qn, bn = q.numpy(), bs.numpy()
    for m in (1, 16, 128):
        ab = synth.bf16_bits(synth.bf16_activations(m, k, seed=1))
        dt = timed(lambda: oracle.nvfp4_matmul(ab, qn, bn, s2))
        key = "nvfp4_gemv_m1" if m == 1 else f"nvfp4_gemm_m{m}"
        if m < 128:
            out[key] = {"value": round(nvfp4_bytes(m, n, k) / dt / 1e9, 3), "unit": "GB/s",
                        "sample": f"the full product, {dt:.2f} s"}
        else:
            out[key] = {"value": round(2 * m * n * k / dt / 1e12, 5), "unit": "TFLOP/s",
                        "sample": f"the full product, {dt:.2f} s"}
    n2, rows = 14336, 16
    codes, sc = synth.fp8_weight(n2, k, seed=0)
    ab = synth.bf16_bits(synth.bf16_activations(rows, k, seed=1))
    cn = codes.numpy()
    dt = timed(lambda: oracle.fp8_matmul(ab, cn, sc))
    out["fp8_gemm_m2048"] = {"value": round(2 * rows * n2 * k / dt / 1e12, 5), "unit": "TFLOP/s",
                             "sample": f"{rows} of the 2048 rows against the full weight, {dt:.2f} s"}
    qb, sb = synth.int8_weight(n2, k, seed=0)
    xb = synth.bf16_bits(synth.bf16_activations(rows, k, seed=1))
    qbn, sbn = qb.numpy(), sb.numpy()

    def w8a8():
        qa, sa = oracle.int8_quantize_rows(xb)
        oracle.int8_matmul(qa, qbn, sa, sbn)

    dt = timed(w8a8)
    out["int8_w8a8_m2048"] = {"value": round(2 * rows * n2 * k / dt / 1e12, 5), "unit": "TFLOP/s",
                              "sample": f"quantize + product of {rows} of the 2048 rows, {dt:.2f} s"}
    stack, scales = synth.fp8_expert_stack(8, n2, k, seed=0)
    offs, ids, _ = synth.moe_routing(4096, seed=2)
    a_moe = synth.bf16_bits(synth.bf16_activations(4096, k, seed=1))
    o = offs.numpy()
    sample_rows = np.concatenate([np.arange(o[z], min(o[z] + 8, o[z + 1])) for z in (0, 1)])
    st, scn, idn = stack.numpy(), scales.numpy(), ids.numpy()
    dt = timed(lambda: oracle.fp8_grouped_matmul(a_moe, st, o, idn, scn, rows=sample_rows))
    out["fp8_grouped_moe"] = {"value": round(2 * len(sample_rows) * n2 * k / dt / 1e12, 5),
                              "unit": "TFLOP/s",
                              "sample": f"{len(sample_rows)} rows of the first two groups "
                                        f"(experts 0, 1), {dt:.2f} s"}
    for v in out.values():
        v["cores"] = cpu_threads()
        v["kind"] = "oracle"
    return out


def run_reference(args, rank, local, world):
    """--impl reference: the CPU oracle on the headline workload and metric."""
    if rank != 0:
        return
    import oracle
    import synth
    inputs = []
    for n, k in GEMV_SHAPES:
        codes, s = synth.fp8_weight(n, k, seed=0)
        x = synth.bf16_activations(1, k, seed=1).reshape(-1)
        inputs.append((codes.numpy(), s, synth.bf16_bits(x)))
    step_bytes = sum(fp8_gemv_bytes(n, k) for n, k in GEMV_SHAPES)
    steps = max(1, min(args.steps, 5))
    warm = min(args.warmup, 1)
    for _ in range(warm):
        for codes, s, xb in inputs:
            oracle.fp8_gemv(xb, codes, s)
    t0 = time.perf_counter()
    for _ in range(steps):
        for codes, s, xb in inputs:
            oracle.fp8_gemv(xb, codes, s)
    dt = time.perf_counter() - t0
    value = step_bytes * steps / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": dt * 1e3 / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": "FP8 W8A16 decode GEMV, M=1, (N,K) in {(4096,4096),"
                               "(14336,4096),(4096,14336)}, bf16 out, per-tensor scale folded",
                   "step": "one GEMV per shape"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cpu_threads(),
                         "kind": "oracle",
                         "sample": f"{steps} step(s) (capped at 5 so the run stays short) of "
                                   "the three decode shapes"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the FP8 GEMV headline (no sub-benchmarks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overlap-weight-reads", action="store_true",
                    help="GEMVs overlap their weight reads with the previous kernel "
                         "(GQ_LAUNCH_OVERLAP_WEIGHT_READS; weights are not written between launches)")
    ap.add_argument("--only", choices=["nvfp4", "gemm", "grouped", "w8a8", "gemv-shapes"], default=None,
                    help="run one sub-benchmark alone and print its result (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, local, world = dist_info()
    if args.impl == "reference":
        run_reference(args, rank, local, world)
        return
    if args.only:
        run_only(args, local)
        return
    run_ours(args, rank, local, world)


def gemv_shape_times(gq, dev, stream, steps, warm):
    """Per-launch time of each FP8 decode shape alone (rotating weight copies)."""
    import synth
    out = {}
    for n, k in GEMV_SHAPES:
        codes, s = synth.fp8_weight(n, k, seed=0)
        x = synth.bf16_activations(1, k, seed=1).reshape(-1).to(dev)
        copies = n_copies(n * k)
        ws = [codes.to(dev) for _ in range(copies)]
        y = torch.empty(n, dtype=torch.bfloat16, device=dev)

        def step(i, ws=ws, x=x, y=y, s=s):
            gq.fp8_gemv(x, ws[i % copies], s, out=y, stream=stream)

        ms = graph_timer(step, steps, warm, min(steps, 200), stream, 1)
        t = ms * 1e-3 / steps
        out[f"{n}x{k}"] = {"us": round(t * 1e6, 3), "GB/s": round(fp8_gemv_bytes(n, k) / t / 1e9, 1)}
        del ws
    return out


def run_only(args, local):
    import gemm_fp8_nvfp4_gb300 as gq
    global STATUS_CHECK
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gq.load_library()
    STATUS_CHECK = gq.device_status
    stream = torch.cuda.Stream(device=dev)
    if args.overlap_weight_reads:
        gq.set_launch_flags(gq.GQ_LAUNCH_OVERLAP_WEIGHT_READS)
    if args.only == "gemv-shapes":
        print(json.dumps({"only": args.only,
                          "shapes": gemv_shape_times(gq, dev, stream, args.steps, args.warmup)}),
              flush=True)
        return
    subs = run_subs(args, gq, dev, stream, measured_peaks(), 1, only=args.only)
    print(json.dumps({"only": args.only, "sub": subs}), flush=True)


if __name__ == "__main__":
    main()
