#!/usr/bin/env python3
"""Benchmark of the block-scaled FP8 linear layer on GB300.

Headline step (one pass of the W8A8 hot path over one batch): per-token 1x128
activation quantisation + block-scaled W8A8 GEMM for the o_proj shape
N = K = 4096 at M = 4096 tokens, with inputs resident in HBM.  Inputs and
weights are rotated over enough copies that every step reads them from HBM
(the rotated set is larger than twice the L2 cache).

One JSON line on stdout (rank 0).  `--sweep` additionally times every
workload shape (W8A8 o_proj / prefill, W8A16 decode and UE8M0) with CUDA-graph
replays over rotated weights and writes the table as JSON to the given path.

`--impl reference` times the float64 CPU oracle on a bounded row sample of the
same workload (the oracle is the only reference implementation there is).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU oracle uses numpy's BLAS; pin its thread count to the cores we have
# so the reported core count is the one used.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

METRIC = "block-FP8 GEMM TFLOP/s (M≥256), weight GB/s (M≤16); % of GB300 roofline"
HEAD_M, HEAD_N, HEAD_K = 4096, 4096, 4096
WORKLOAD = "W8A8 o_proj linear, N=K=4096, M=4096: act quant (1x128) + block-scaled GEMM"
FP8_PER_BF16 = 2.0       # nominal dense fp8 : bf16 tensor rate (4.5 / 2.25 PFLOP/s)

# DRAM traffic of one w8a8_pair_kernel launch at M = N = K = 4096, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), valid only for
# the kernel source it was taken on: reported as null once that file changes.
TRAFFIC_CAPTURE = {"source": "block_scaled_fp8_bf16_gb300/csrc/gemm_w8a8_pair.cu",
                   "md5": "135012a15c3e9628750e7aad167ee5e5",
                   "bytes": 34_142_976 + 2_013_184}


def measured_traffic():
    import hashlib
    path = os.path.join(ROOT, TRAFFIC_CAPTURE["source"])
    try:
        with open(path, "rb") as f:
            digest = hashlib.md5(f.read()).hexdigest()
    except OSError:
        return None
    return TRAFFIC_CAPTURE["bytes"] if digest == TRAFFIC_CAPTURE["md5"] else None


def peaks():
    p = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
    if "hbm_gbs" in p and "bf16_tflops" in p:
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling in the background; each line is stamped with the
    host time it arrived so that only samples inside the timed region count."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.dev = device_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(0.5)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(2 * self.period / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        window = [l for t, l in self.lines if self.t0 is not None and self.t0 <= t <= (self.t1 or t)]
        if not window:     # region shorter than one sampling period: take the first sample after it began
            window = [l for t, l in self.lines if self.t0 is not None and t >= self.t0][:1]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="gloo")
    return world, rank, local


def dist_max(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- GPU arm

def _rot_copies(bytes_per_copy: int, l2_bytes: int, cap: int = 64) -> int:
    need = 2 * l2_bytes
    return max(2, min(cap, -(-need // max(1, bytes_per_copy))))


def build_w8a8_set(M, N, K, copies, seed=0, outliers=True):
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    from synth import torch_gen as tg
    x0 = tg.activations(seed, M, K, outliers=outliers)
    w0 = tg.weights_bf16(seed, N, K)
    b0, bs0 = fp8blk.quant_weight(w0)
    del w0
    sets = []
    lds = fp8blk.act_scales_pitch(M)
    for _ in range(copies):
        sets.append({
            "x": x0.clone(), "b": b0.clone(), "bs": bs0.clone(),
            "a": torch.empty((M, K), dtype=torch.uint8, device="cuda"),
            "s": torch.empty((K // 128, lds), dtype=torch.float32, device="cuda"),
            "c": torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
        })
    return sets


def gpu_arm(args, world, rank, local):
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    M, N, K = HEAD_M, HEAD_N, HEAD_K
    per_copy = M * K * 2 + M * K + N * K + M * N * 2 + (K // 128) * M * 4
    R = _rot_copies(per_copy, l2)
    sets = build_w8a8_set(M, N, K, R)
    stream = torch.cuda.current_stream()

    # One step: the quantiser, then the GEMM launched with programmatic
    # dependent launch (it starts streaming the weights while the quantiser
    # finishes, and waits for it before reading the codes and scales).
    pdl = fp8blk.FLAG_PDL

    def step(i):
        s = sets[i % R]
        fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"], stream)
        fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"], stream, flags=pdl)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if fp8blk.fp8blk_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # Timed region: K steps between two events on the launching stream, with
    # nothing recorded between a step's two kernels.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    dist_barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    clocks.mark_start()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop()
    dist_barrier(world)
    ms_total = dist_max(ev0.elapsed_time(ev1), world)
    err = fp8blk.fp8blk_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    # Roofline of the dominant kernel (the GEMM), timed in its own pass right
    # after: the same K launches over the same rotated sets, each between two
    # events on the launching stream, launched plainly so that each event
    # pair brackets exactly one GEMM.
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        s = sets[i % R]
        g0[i].record(stream)
        fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"], stream)
        g1[i].record(stream)
    torch.cuda.synchronize()
    gemm_ms = dist_max(sum(a.elapsed_time(b) for a, b in zip(g0, g1)) / args.steps, world)

    flop = 2.0 * M * N * K
    ms_step = ms_total / args.steps
    value = world * flop / (ms_step * 1e-3) / 1e12
    pk = peaks()
    fp8_peak = pk["bf16"] * FP8_PER_BF16
    achieved = flop / (gemm_ms * 1e-3) / 1e12

    # End to end through the C ABI from pinned host buffers: every step copies
    # its activations host -> device, runs quant + GEMM and copies C back,
    # all inside the timed region.  The copies run on their own streams so
    # that step i's H2D and step i-1's D2H overlap step i's kernels (a
    # serving loop pipelines its transfers the same way); events order every
    # reuse of a rotated buffer set.
    e2e_steps = max(3, min(args.steps, 100))
    xh = [sets[i]["x"].cpu().pin_memory() for i in range(R)]
    ch = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n, e_start=None, e_stop=None):
        ev_in = [torch.cuda.Event() for _ in range(R)]
        ev_comp = [torch.cuda.Event() for _ in range(R)]
        ev_out = [torch.cuda.Event() for _ in range(R)]
        if e_start is not None:
            e_start.record(stream)
            s_in.wait_event(e_start)
            s_out.wait_event(e_start)
        for i in range(n):
            j = i % R
            s = sets[j]
            if i >= R:
                s_in.wait_event(ev_comp[j])          # step i - R has read x[j]
            with torch.cuda.stream(s_in):
                s["x"].copy_(xh[j], non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if i >= R:
                stream.wait_event(ev_out[j])         # step i - R's C[j] has left the device
            fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"], stream)
            fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"], stream, flags=pdl)
            ev_comp[j].record(stream)
            s_out.wait_event(ev_comp[j])
            with torch.cuda.stream(s_out):
                ch[i % 2].copy_(s["c"], non_blocking=True)
            ev_out[j].record(s_out)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)
        if e_stop is not None:
            e_stop.record(stream)

    e2e_run(2 * R)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1), world) / e2e_steps
    e2e_value = world * flop / (e2e_ms * 1e-3) / 1e12

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (bf16 in/out)",
        "data": "synthetic (seeded torch generators: x ~ N(0,1) with 1% outlier channels x20, w ~ N(0,0.02))",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                   "l2": f"inputs rotated over {R} copies ({R * per_copy / 2**20:.0f} MiB > 2x L2 {l2 / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "w8a8_pair_kernel (block-scaled e4m3 GEMM, CTA pairs)",
                     "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4),
                     "peak_note": f"{pk['source']} bf16 burst {pk['bf16']} TFLOP/s x {FP8_PER_BF16} (nominal fp8:bf16)",
                     "gemm_us": round(gemm_ms * 1e3, 2), "traffic": measured_traffic(),
                     "timing": "K plain GEMM launches over the same rotated sets right after the timed region, "
                               "each between two events on the launching stream (the timed steps launch the "
                               "GEMM with programmatic dependent launch and record nothing between kernels)",
                     "traffic_note": "DRAM bytes per launch from one ncu capture of this kernel source; "
                                     "algorithmic reads A+As+B+Bs = 34.08 MB, C stays in L2"},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2, "steps": e2e_steps,
                "note": "pinned host buffers; H2D and D2H on their own streams, overlapping neighbouring steps"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    return line


# ---------------------------------------------------------------- CPU oracle

def oracle_linear_sample(rows: int, seed: int = 0):
    """Inputs for the oracle leg: the same workload (N = K = 4096) on a seeded
    row sample.  Weight quantisation is input preparation, not timed."""
    import numpy as np

    import oracle
    import synth
    x = synth.activations(seed, HEAD_M, HEAD_K, outliers=True)
    idx = synth.sample_rows(seed, HEAD_M, rows)
    b, bs = oracle.quant_weight_128x128(synth.weights_bf16(seed, HEAD_N, HEAD_K))
    return np.ascontiguousarray(x[idx]), b, bs


def oracle_step(xs, b, bs):
    import oracle
    a, s = oracle.quant_act_1x128(xs)
    return oracle.gemm_w8a8(a, s, b, bs)


def cpu_baseline(rows: int = 64, min_seconds: float = 10.0):
    xs, b, bs = oracle_linear_sample(rows)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(xs, b, bs)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or n >= 200:
            break
    per = dt / n
    value = 2.0 * rows * HEAD_N * HEAD_K / per / 1e12
    return {"value": round(value, 6), "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{rows} seeded rows of the M=4096 o_proj batch (N=K=4096), act quant + W8A8 product in "
                      f"float64 numpy, {n} repetitions over {dt:.1f} s"}


def reference_arm(args, world, rank):
    if rank != 0:
        return None
    rows = 64
    xs, b, bs = oracle_linear_sample(rows)
    for _ in range(args.warmup):
        oracle_step(xs, b, bs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(xs, b, bs)
    dt = time.perf_counter() - t0
    per = dt / args.steps
    value = 2.0 * rows * HEAD_N * HEAD_K / per / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy generators)",
        "config": {"workload": WORKLOAD, "M": HEAD_M, "N": HEAD_N, "K": HEAD_K,
                   "sample": f"{rows} rows per step", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
                         "sample": f"{rows} seeded rows of the M=4096 batch per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def graph_time(calls, reps=10):
    """Median time per call (us) of `calls` captured once in a CUDA graph and
    replayed `reps` times (three untimed replays first); raises if a kernel
    set the library's device error word."""
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in calls:
            c()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / len(calls))
    if fp8blk.fp8blk_device_error() != 0:
        raise RuntimeError("device error word set")
    return statistics.median(times) * 1e3     # us per call


# ---------------------------------------------------------------- sweep

def sweep(out_path, kinds=None):
    """Times every workload shape with CUDA-graph replays over rotated copies
    (kinds: optional subset of "w8a8", "grouped", "w8a16", "linear", "mx")."""
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    from synth import torch_gen as tg
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    pk = peaks()
    rows = []

    def record(kind, M, N, K, us, flop, bytes_, tensor_peak):
        t_tensor = flop / (tensor_peak * 1e12)
        t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
        roof_us = max(t_tensor, t_hbm) * 1e6
        rows.append({"kind": kind, "M": M, "N": N, "K": K, "us": round(us, 3),
                     "tflops": round(flop / (us * 1e-6) / 1e12, 2),
                     "weight_gbs": round(N * K / (us * 1e-6) / 1e9, 1),
                     "bytes_gbs": round(bytes_ / (us * 1e-6) / 1e9, 1),
                     "bound": "tensor" if t_tensor >= t_hbm else "hbm",
                     "roofline_frac": round(roof_us / us, 4)})
        print(json.dumps(rows[-1]), file=sys.stderr)

    fp8_peak = pk["bf16"] * FP8_PER_BF16
    # W8A8: o_proj and prefill shapes (GEMM alone, and quant+GEMM)
    w8a8 = [(M, 4096, 4096) for M in (1, 16, 128, 1024, 4096)] + [(16, 256, 512)]
    for M in (256, 2048, 8192):
        for N, K in ((7168, 2048), (2048, 7168), (18432, 7168), (7168, 18432)):
            w8a8.append((M, N, K))
    if kinds is not None and "w8a8" not in kinds:
        w8a8 = []
    PDL = fp8blk.FLAG_PDL
    for M, N, K in w8a8:
        per = M * K * 3 + N * K + M * N * 2
        R = _rot_copies(per, l2, cap=32)
        sets = build_w8a8_set(M, N, K, R, outliers=(N == 4096 and K == 4096))
        for s in sets:
            fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"])
        byt = M * K + (K // 128) * M * 4 + N * K + (N // 128) * (K // 128) * 4 + 2 * M * N
        for flags, tag in ((0, ""), (PDL, "_pdl")):
            calls = [lambda s=s, f=flags: fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"], flags=f)
                     for s in sets]
            record("w8a8_gemm" + tag, M, N, K, graph_time(calls), 2.0 * M * N * K, byt, fp8_peak)
            calls2 = [lambda s=s, f=flags: (fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"]),
                                            fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"],
                                                                    flags=f)) for s in sets]
            record("w8a8_linear" + tag, M, N, K, graph_time(calls2), 2.0 * M * N * K, byt + 2 * M * K, fp8_peak)
            if M <= fp8blk.LINEAR_FUSED_MAX_M:
                calls3 = [lambda s=s, f=flags: fp8blk.fp8blk_linear_w8a8(s["x"], s["b"], s["bs"], s["c"], flags=f)
                          for s in sets]
                record("w8a8_linear_fused" + tag, M, N, K, graph_time(calls3), 2.0 * M * N * K,
                       byt + 2 * M * K - M * K - (K // 128) * M * 4, fp8_peak)
        qcalls = [lambda s=s: fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"]) for s in sets]
        record("quant_act", M, 0, K, graph_time(qcalls), 0.0, 3 * M * K + (K // 128) * M * 4, fp8_peak)
        del sets
        torch.cuda.empty_cache()
    # Grouped (mixture-of-experts) W8A8: G experts with the same number of
    # 128-row tiles each, N x K weights per expert.
    grouped = [(8, 512, 4096, 4096), (32, 256, 2048, 7168), (64, 128, 7168, 2048)]
    if kinds is not None and "grouped" not in kinds:
        grouped = []
    for G, per_group, N, K in grouped:
        M = G * per_group
        xg = tg.activations(1, M, K)
        a, sc = fp8blk.quant_act(xg)
        ws = [fp8blk.quant_weight(tg.weights_bf16(1 + e, N, K)) for e in range(G)]
        b = torch.stack([w[0] for w in ws])
        bs = torch.stack([w[1] for w in ws])
        del ws
        rg = torch.arange(G, dtype=torch.int32, device="cuda").repeat_interleave(per_group)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        calls = [lambda: fp8blk.fp8blk_gemm_w8a8_grouped(a, sc, b, bs, rg, c)]
        byt = M * K + (K // 128) * M * 4 + G * N * K + G * (N // 128) * (K // 128) * 4 + 2 * M * N
        record(f"w8a8_grouped_G{G}", M, N, K, graph_time(calls * 4), 2.0 * M * N * K, byt, fp8_peak)
        del a, sc, b, bs, c
        torch.cuda.empty_cache()
    # W8A16 fp32-scale decode and UE8M0
    w8a16 = []
    for N, K in ((4096, 4096), (28672, 4096), (4096, 14336)):
        for M in (1, 2, 4, 8, 16):
            w8a16.append((0, M, N, K))
    for N, K in ((2048, 7168), (7168, 2048)):
        for M in (1, 4, 16, 32, 128, 512, 4096):
            w8a16.append((1, M, N, K))
    if kinds is not None and "w8a16" not in kinds:
        w8a16 = []
    for fmt, M, N, K in w8a16:
        per = N * K + M * K * 2 + M * N * 2
        R = _rot_copies(per, l2, cap=64)
        x = tg.activations(1, M, K)
        if fmt == 0:
            b, bs = fp8blk.quant_weight(tg.weights_bf16(1, N, K))
        else:
            b, bs = tg.ue8m0_weights(1, N, K)
        sets = [(x.clone(), b.clone(), bs.clone(), torch.empty((M, N), dtype=torch.bfloat16, device="cuda"))
                for _ in range(R)]
        fn = fp8blk.fp8blk_gemv_w8a16 if M <= 16 else fp8blk.fp8blk_gemm_w8a16
        sc_bytes = (N // 128) * (K // 128) * 4 if fmt == 0 else (N // 32) * (K // 32)
        byt = N * K + sc_bytes + M * K * 2 + M * N * 2
        for flags, tag in ((0, ""), (PDL, "_pdl")):
            calls = [lambda s=s, f=flags: fn(s[0], s[1], s[2], fmt, s[3], flags=f) for s in sets]
            record(("w8a16_f32" if fmt == 0 else "w8a16_ue8m0") + tag, M, N, K, graph_time(calls),
                   2.0 * M * N * K, byt, pk["bf16"])
        del sets
        torch.cuda.empty_cache()
    # Decode-size W8A8 linear: the fused quantising kernel against
    # fp8blk_quant_act + fp8blk_gemm_w8a8 (the rows the binding's choice
    # between the two forms is taken from).
    linear = [(M, N, K) for M in (2, 4, 8, 16, 32) for N, K in ((4096, 4096), (7168, 2048), (2048, 7168), (256, 512))]
    if kinds is not None and "linear" not in kinds:
        linear = []
    for M, N, K in linear:
        per = M * K * 3 + N * K + M * N * 2
        R = _rot_copies(per, l2, cap=64)
        sets = build_w8a8_set(M, N, K, R, outliers=False)
        byt = N * K + (N // 128) * (K // 128) * 4 + 2 * M * K + 2 * M * N
        for flags, tag in ((0, ""), (PDL, "_pdl")):
            two = [lambda s=s, f=flags: (fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"]),
                                         fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"], flags=f))
                   for s in sets]
            record("w8a8_linear" + tag, M, N, K, graph_time(two), 2.0 * M * N * K, byt, fp8_peak)
            fused = [lambda s=s, f=flags: fp8blk.fp8blk_linear_w8a8(s["x"], s["b"], s["bs"], s["c"], flags=f)
                     for s in sets]
            record("w8a8_linear_fused" + tag, M, N, K, graph_time(fused), 2.0 * M * N * K, byt, fp8_peak)
        del sets
        torch.cuda.empty_cache()
    # W8A8 in the 32x32 UE8M0 format (block-scaled tensor cores): the product
    # alone and quantiser + product.
    mx = [(M, N, K) for M in (128, 512, 4096, 8192) for N, K in ((2048, 7168), (7168, 2048))]
    if kinds is not None and "mx" not in kinds:
        mx = []
    for M, N, K in mx:
        per = M * K * 3 + N * K + M * N * 2
        R = _rot_copies(per, l2, cap=32)
        x = tg.activations(1, M, K)
        b, eb = tg.ue8m0_weights(1, N, K)
        bsf = fp8blk.ue8m0_weight_sf(eb)     # offline: the weight exponents in the tiled scale layout
        sets = []
        for _ in range(R):
            a, e = fp8blk.quant_act_ue8m0(x)
            sets.append({"x": x.clone(), "a": a, "e": e, "b": b.clone(), "eb": bsf.clone(),
                         "c": torch.empty((M, N), dtype=torch.bfloat16, device="cuda")})
        byt = M * K + e.numel() + N * K + bsf.numel() + 2 * M * N
        calls = [lambda s=s: fp8blk.fp8blk_gemm_w8a8_ue8m0(s["a"], s["e"], s["b"], s["eb"], s["c"]) for s in sets]
        record("w8a8_ue8m0_gemm", M, N, K, graph_time(calls), 2.0 * M * N * K, byt, fp8_peak)
        calls = [lambda s=s: (fp8blk.fp8blk_quant_act_ue8m0(s["x"], s["a"], s["e"]),
                              fp8blk.fp8blk_gemm_w8a8_ue8m0(s["a"], s["e"], s["b"], s["eb"], s["c"],
                                                            flags=PDL)) for s in sets]
        record("w8a8_ue8m0_linear_pdl", M, N, K, graph_time(calls), 2.0 * M * N * K, byt + 2 * M * K, fp8_peak)
        del sets
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump({"peaks": pk, "fp8_peak": fp8_peak, "rows": rows}, f, indent=1)


# ---------------------------------------------------------------- profiling cases

def run_case(spec: str, iters: int):
    """Runs one kernel configuration `iters` times, untimed (for ncu captures).
    spec: w8a8:M,N,K | quant:M,K | w8a16:M,N,K,fmt | linear:M,N,K (fused quantising
    W8A8, M <= 32) | grouped:G,rows_per_group,N,K | mx:M,N,K (UE8M0 W8A8:
    quantiser + block-scaled product)"""
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    from synth import torch_gen as tg
    kind, dims = spec.split(":")
    v = [int(t) for t in dims.split(",")]
    if kind in ("w8a8", "quant"):
        if kind == "w8a8":
            M, N, K = v
        else:
            (M, K), N = v, 128
        s = build_w8a8_set(M, N, K, 1)[0]
        for _ in range(iters):
            fp8blk.fp8blk_quant_act(s["x"], s["a"], s["s"])
            if kind == "w8a8":
                fp8blk.fp8blk_gemm_w8a8(s["a"], s["s"], s["b"], s["bs"], s["c"])
    elif kind == "linear":
        M, N, K = v
        x = tg.activations(1, M, K)
        b, bs = fp8blk.quant_weight(tg.weights_bf16(1, N, K))
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(iters):
            fp8blk.fp8blk_linear_w8a8(x, b, bs, c)
    elif kind == "grouped":
        G, rows_per_group, N, K = v
        M = G * rows_per_group
        a, sc = fp8blk.quant_act(tg.activations(1, M, K))
        ws = [fp8blk.quant_weight(tg.weights_bf16(1 + e, N, K)) for e in range(G)]
        b = torch.stack([w[0] for w in ws])
        bs = torch.stack([w[1] for w in ws])
        rg = torch.arange(G, dtype=torch.int32, device="cuda").repeat_interleave(rows_per_group)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(iters):
            fp8blk.fp8blk_gemm_w8a8_grouped(a, sc, b, bs, rg, c)
    elif kind == "mx":
        M, N, K = v
        x = tg.activations(1, M, K)
        b, eb = tg.ue8m0_weights(1, N, K)
        bsf = fp8blk.ue8m0_weight_sf(eb)
        a, e = fp8blk.quant_act_ue8m0(x)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(iters):
            fp8blk.fp8blk_quant_act_ue8m0(x, a, e)
            fp8blk.fp8blk_gemm_w8a8_ue8m0(a, e, b, bsf, c)
    elif kind == "w8a16":
        M, N, K, fmt = v
        x = tg.activations(1, M, K)
        if fmt == 0:
            b, bs = fp8blk.quant_weight(tg.weights_bf16(1, N, K))
        else:
            b, bs = tg.ue8m0_weights(1, N, K)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(iters):
            fp8blk.fp8blk_gemm_w8a16(x, b, bs, fmt, c)
    else:
        raise SystemExit(f"unknown case {spec}")
    torch.cuda.synchronize()
    if fp8blk.fp8blk_device_error() != 0:
        raise SystemExit("device error word set")


# ---------------------------------------------------------------- probe

def probe():
    """Memory-system figures that frame the rooflines: device read, write and
    copy rates by size with torch reductions, fills and copies, the library's
    plain streaming-read kernel on the weight-set sizes of the decode-size
    workloads, and the host link's copy-engine rates for
    one 33.5 MB transfer (the headline step's activations or output), alone
    and with both directions at once.  One JSON line per measurement."""
    import torch
    dev = torch.device("cuda:0")

    def best(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        t = 1e9
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t = min(t, a.elapsed_time(b) * 1e-3)
        return t

    for nbytes in (1 << 27, 1 << 29, 1 << 31):
        a = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
        b = torch.empty_like(a)
        for what, fn, moved in (("read (sum)", lambda: a.sum(), nbytes), ("write (fill)", lambda: b.fill_(1.0), nbytes),
                                ("copy (read + write)", lambda: b.copy_(a), 2 * nbytes)):
            t = best(fn)
            print(json.dumps({"probe": "hbm", "op": what, "mib": nbytes >> 20, "gb_s": round(moved / t / 1e9, 1)}))
        del a, b
    # The library's plain streaming-read kernel on the decode-size weight-set
    # sizes, in CUDA-graph replays over rotated copies larger than 2x L2 (as
    # the sweep times the GEMMs): the rate that any kernel reading a weight
    # set of that size once can reach.
    import block_scaled_fp8_bf16_gb300 as fp8blk
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    for what, nbytes in (("2048x7168 codes", 2048 * 7168), ("4096x4096 codes", 4096 * 4096),
                         ("4096x14336 codes", 4096 * 14336), ("28672x4096 codes", 28672 * 4096),
                         ("512 MiB", 1 << 29)):
        reps = max(2, -(-(1 << 28) // nbytes))
        bufs = [torch.full((nbytes,), i, dtype=torch.uint8, device=dev) for i in range(reps)]
        us = graph_time([lambda b=b: fp8blk.fp8blk_debug_stream_read(b, sink) for b in bufs])
        print(json.dumps({"probe": "hbm, plain read kernel (fp8blk_debug_stream_read), CUDA graph", "op": what,
                          "mb": round(nbytes / 1e6, 1), "us": round(us, 2), "gb_s": round(nbytes / us / 1e3, 1)}))
        del bufs
    # Per-kernel floor: a one-element kernel replayed 200 times in a CUDA graph.
    t1 = torch.zeros(1, device=dev)
    g = torch.cuda.CUDAGraph()
    s_cap = torch.cuda.Stream()
    s_cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_cap):
        t1.add_(1.0)
    torch.cuda.current_stream().wait_stream(s_cap)
    with torch.cuda.graph(g, stream=s_cap):
        for _ in range(200):
            t1.add_(1.0)
    t = best(g.replay) / 200
    print(json.dumps({"probe": "kernel floor", "op": "one-element kernel, 200 per CUDA graph", "us_per_kernel":
                      round(t * 1e6, 2)}))
    n = HEAD_M * HEAD_K * 2
    h = [torch.empty(n, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    cur = torch.cuda.current_stream()

    def both():
        ev = torch.cuda.Event()
        ev.record(cur)
        for s, dst, src in ((s_in, d[0], h[0]), (s_out, h[1], d[1])):
            s.wait_event(ev)
            with torch.cuda.stream(s):
                dst.copy_(src, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    for what, fn in (("h2d", lambda: d[0].copy_(h[0], non_blocking=True)),
                     ("d2h", lambda: h[1].copy_(d[1], non_blocking=True)),
                     ("h2d + d2h at once (per direction)", both)):
        t = best(fn)
        print(json.dumps({"probe": "host link, pinned, copy engines", "op": what, "mb": round(n / 1e6, 1),
                          "gb_s": round(n / t / 1e9, 1)}))


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--sweep", default=None, metavar="OUT.json",
                    help="also time every workload shape and write the table to OUT.json")
    ap.add_argument("--sweep-kinds", default=None,
                    help="comma list restricting --sweep to some of: w8a8, grouped, w8a16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None, help="run one configuration untimed (w8a8:M,N,K | quant:M,K | "
                    "linear:M,N,K | grouped:G,rows,N,K | mx:M,N,K | "
                    "w8a16:M,N,K,fmt) for profiling")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--probe", action="store_true",
                    help="print device-memory and host-link rates (torch operations only) and exit")
    args = ap.parse_args()
    if args.probe:
        probe()
        return
    if args.case:
        import block_scaled_fp8_bf16_gb300 as fp8blk
        fp8blk._L()
        run_case(args.case, args.iters)
        return
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup()

    if args.impl == "reference":
        line = reference_arm(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import block_scaled_fp8_bf16_gb300 as fp8blk
    fp8blk._L()
    line = gpu_arm(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline()
        if args.sweep:
            os.makedirs(os.path.dirname(os.path.abspath(args.sweep)), exist_ok=True)
            sweep(args.sweep, None if args.sweep_kinds is None else set(args.sweep_kinds.split(",")))
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
