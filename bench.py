"""Benchmark of the affine group-wise quantized matmul library on GB300.

One step is the decode GEMV (qmv) over the decode workload: K=5120 N=17408
and K=17408 N=5120, each with 4-bit and 8-bit codes (group 64, bf16 scales
and biases, W ~ N(0, 0.02) quantized with scale=(max-min)/(2^bits-1),
bias=min, x ~ N(0, 1)).  ``value`` is the whole-job achieved HBM bandwidth
over algorithmic bytes (codes + scales + biases + x + y) in GB/s.  Each
case keeps two copies of its inputs and alternates between them, so the
working set of a step pass (580 MB) is larger than the 129 MB L2.

The same JSON line carries, measured after the main timed region and with
their own rotation: the prefill GEMM (M=600, K=5120, N=17408), the M sweep
at K=N=5120, the sorted-MoE gather (E=128, top_k=8, 573 tokens; K=2816
N=704 and K=704 N=2816) and the 4-bit vs 8-bit controlled pair, each with
its binding roofline.

``--impl reference`` times the f64 CPU checker on the same metric (the
slow reference program, not a target).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

STEPS_PER_GRAPH = 20

METRIC = "qmv HBM GB/s and qmm/gather_qmm TFLOPS on 1 GB300, % of roofline"
DECODE_CASES = [(5120, 17408, 4), (5120, 17408, 8), (17408, 5120, 4), (17408, 5120, 8)]
WORKLOAD = ("qmv decode M=1: K=5120 N=17408 and K=17408 N=5120, 4-bit and 8-bit, group 64, "
            "bf16 scales/biases")
# the same config dict on both arms
CONFIG = {"workload": WORKLOAD, "M": 1, "group_size": 64,
          "l2": "inputs larger than L2: each case alternates two input copies "
                "(580 MB working set vs 129 MB L2)",
          "parallelism": "replicas (one per GPU, no collective)"}
PREHEAT_S = 0.3


def qmv_bytes(K, N, bits, group=64):
    return N * K * bits // 8 + N * (K // group) * 4 + K * 2 + N * 2


def qmm_bytes(M, K, N, bits, group=64):
    return N * K * bits // 8 + N * (K // group) * 4 + M * K * 2 + M * N * 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ helpers

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "qmv_stream_decode_traffic.txt")
QMV_SOURCES = [os.path.join(ROOT, "affine_bit_matmul_gb300", "csrc", f)
               for f in ("qmv.cu", "mxq_device.cuh")]


def qmv_source_hash():
    import hashlib

    h = hashlib.sha256()
    for f in QMV_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_per_launch():
    """DRAM bytes (read + write) per qmv launch, mean over the four decode
    cases, from the committed ncu capture; None when the kernel sources have
    changed since that capture (or there is none)."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_hash") != qmv_source_hash():
            return None
        return int(fields["mean_dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None



class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons every 20 ms.

    ``mark()`` returns the current sample count, so that ``summary(a, b)``
    can describe the samples taken between two marks (one window per
    measured entry)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        self.rows = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        self.file.flush()
        with open(self.file.name) as f:
            text = f.read()
        out = []
        for line in text.splitlines():
            r = line.strip().split(",")
            try:
                reasons = {n for n, v in zip(self.NAMES, r[5:9]) if v.strip().lower() == "active"}
                out.append((float(r[1]), float(r[2]), float(r[3]), reasons))
            except (ValueError, IndexError):
                continue
        return out

    def mark(self):
        if self.proc is None:
            return 0
        time.sleep(0.05)  # let the sampler write what it has seen so far
        return len(self._read())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.rows = self._read()
        os.unlink(self.file.name)

    def summary(self, a=0, b=None):
        rows = (self.rows if self.rows is not None else self._read())[a:b]
        if not rows:
            return None
        lo, hi = min(r[2] for r in rows), max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= (lo + hi) / 2] or rows  # samples drawing power
        reasons = sorted(set().union(*[r[3] for r in rows]))
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": hi}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value, world):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ device inputs


def dev_bf16(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(
        torch.bfloat16).to(dev)


def dev_codes(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).to(dev)


class DenseInputs:
    def __init__(self, W, M, K, N, bits, dev, copies, x_seed=1, group=64):
        import torch

        qw = synth.quantize(W, bits, group)
        self.M, self.K, self.N, self.bits, self.group = M, K, N, bits, group
        self.host = (qw.w, qw.scales, qw.biases)
        self.x_host = synth.activations(M, K, seed=x_seed)
        w, s, b = dev_codes(qw.w, dev), dev_bf16(qw.scales, dev), dev_bf16(qw.biases, dev)
        self.copies = [(w, s, b)] + [(w.clone(), s.clone(), b.clone()) for _ in range(copies - 1)]
        self.x = dev_bf16(self.x_host, dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)


# --no-graphs issues every launch directly on the stream (same kernels, same
# arguments); ncu's launch list is taken that way because it does not follow
# launches made during stream capture.
USE_GRAPHS = True


class _Direct:
    """Stands in for a CUDA graph: replay() issues the launches directly."""

    def __init__(self, fn, count):
        self.fn, self.count = fn, count

    def replay(self):
        for i in range(self.count):
            self.fn(i)


def capture(fn, count):
    """A CUDA graph of fn(0), ..., fn(count - 1) (launch overhead out of the
    timed work; inputs alternate between copies by the index)."""
    import torch

    if not USE_GRAPHS:
        return _Direct(fn, count)

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(count):  # warm the code path on the capture stream
            fn(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(count):
            fn(i)
    torch.cuda.synchronize()
    return g


def time_launches(fn, iters, stream, reps=5, preheat_s=0.05):
    """Median per-launch device time of fn over graphs of ``iters`` launches
    (CUDA events on the launching stream around each graph replay), after
    replaying the graph for ``preheat_s`` seconds (untimed: the GPU reaches
    its loaded clocks, and the clock sampler sees the entry)."""
    import torch

    g = capture(fn, iters)
    g.replay()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + preheat_s
    while time.perf_counter() < t_end:
        g.replay()
        torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3 / iters)
    return statistics.median(ts), ts


# ------------------------------------------------------------------ our arm


def run_mxq(args):
    import torch

    import affine_bit_matmul_gb300 as mxq
    from affine_bit_matmul_gb300 import build as _build

    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    hbm, bf16_peak, bf16_sus, peak_src = load_peaks()
    clocks = Clocks(local)
    clocks.start()

    # ---- decode workload: 4 cases, two input copies each
    Ws = {}
    cases = []
    for K, N, bits in DECODE_CASES:
        if (K, N) not in Ws:
            Ws[(K, N)] = synth.dense_weights(N, K, seed=0)
        cases.append(DenseInputs(Ws[(K, N)], 1, K, N, bits, dev, copies=2))
    step_bytes = sum(qmv_bytes(c.K, c.N, c.bits) for c in cases)

    def step(i):
        for c in cases:
            w, s_, b = c.copies[i % 2]
            mxq.qmv(c.x[0], w, s_, b, c.bits, out=c.y[0])

    # graphs of STEPS_PER_GRAPH steps (inputs alternate by step parity) plus
    # one-step graphs per parity for a remainder: exactly args.steps steps run
    # in the timed region
    big = capture(lambda j: step(j), STEPS_PER_GRAPH)
    graphs = [capture(lambda j, par=par: step(par), 1) for par in (0, 1)]

    # per-case device time, each case alone (graphs of 20 launches): the
    # breakdown of the step; it also brings the GPU to its loaded clocks
    per_case = []
    for c in cases:
        m0 = clocks.mark()
        t, _ = time_launches(
            lambda i, c=c: mxq.qmv(c.x[0], *c.copies[i % 2], c.bits, out=c.y[0]), 20, stream,
            reps=25)
        nb = qmv_bytes(c.K, c.N, c.bits)
        per_case.append({"n": "qmv K=%d N=%d b%d g64" % (c.K, c.N, c.bits), "us": r3(t * 1e6),
                         "GBs": r1(nb / t / 1e9), "bound": "hbm", "frac": r4(nb / t / 1e9 / hbm),
                         "mhz": _mhz(clocks.summary(m0))})

    # preheat: the decode step back to back for about PREHEAT_S seconds, so
    # that the timed region starts at the loaded clocks (untimed)
    t_end = time.perf_counter() + PREHEAT_S
    while time.perf_counter() < t_end:
        big.replay()
        torch.cuda.synchronize()
    for i in range(args.warmup):
        graphs[i % 2].replay()
    torch.cuda.synchronize()
    m_timed = clocks.mark()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    full = args.steps // STEPS_PER_GRAPH
    for _ in range(full):
        big.replay()
    for i in range(full * STEPS_PER_GRAPH, args.steps):
        graphs[i % 2].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    local_elapsed = t0.elapsed_time(t1) * 1e-3
    elapsed = max_over_ranks(local_elapsed, world)
    value = step_bytes * args.steps * world / elapsed / 1e9
    # the timed region holds nothing but qmv launches (four per step): the
    # kernel's algorithmic bytes per launch over its mean launch duration
    # there is this rank's step bytes over its time per step
    achieved = step_bytes * args.steps / local_elapsed / 1e9
    m_timed_end = clocks.mark()

    # ---- end to end through the public API with host buffers
    pinned = []
    for c in cases:
        w, s, b = c.host
        pinned.append({
            "w": torch.from_numpy(w.view(np.int32).copy()).pin_memory(),
            "s": torch.from_numpy(s.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
            "b": torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
            "x": torch.from_numpy(c.x_host.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
            "y": torch.empty((c.N,), dtype=torch.bfloat16).pin_memory(),
        })
    h2d = sum(sum(p[k].numel() * p[k].element_size() for k in ("w", "s", "b", "x")) for p in pinned)
    d2h = sum(p["y"].numel() * 2 for p in pinned)

    def e2e_step():
        for c, p in zip(cases, pinned):
            w, s, b = c.copies[0]
            w.copy_(p["w"], non_blocking=True)
            s.copy_(p["s"], non_blocking=True)
            b.copy_(p["b"], non_blocking=True)
            c.x[0].copy_(p["x"][0], non_blocking=True)
            mxq.qmv(c.x[0], w, s, b, c.bits, out=c.y[0])
            p["y"].copy_(c.y[0], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a, bq = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    bq.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_elapsed = max_over_ranks(a.elapsed_time(bq) * 1e-3, world)
    e2e_value = step_bytes * e2e_steps * world / e2e_elapsed / 1e9

    secondary = []
    if not args.no_secondary:
        secondary = secondary_measurements(mxq, dev, stream, hbm, bf16_peak, Ws, clocks)
    clocks.stop()
    clk = clocks.summary(m_timed, m_timed_end)
    # the 20 ms sampler may see no sample inside a short timed region: then
    # the window is widened to the preheat before it, the same launches
    if clk is None or clk["samples"] < 3:
        clk = clocks.summary(0, m_timed_end)
        if clk is not None:
            clk["window"] = "per-case timing, preheat and timed region"
    elif clk is not None:
        clk["window"] = "timed region"

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u4/u8 codes, bf16 x, fp32 accumulate",
        "data": "synthetic (seeded W~N(0,0.02) quantized per the workload recipe, x~N(0,1))",
        "config": CONFIG,
        "roofline": {"bound": "hbm", "kernel": "qmv_stream_kernel (4- and 8-bit)",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic_per_launch(),
                     "algorithmic_bytes_per_launch": step_bytes // len(cases),
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"},
        "gpu_launches": len(cases) * args.steps,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "public API qmv with inputs copied from pinned host memory every step"},
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    # last, so that the end of the line carries the workload's own configs:
    # every other measured entry, then the workload configs (M sweep, 4/8-bit
    # pair, sorted-MoE gather, prefill), then the decode cases of `value`
    line["secondary"] = secondary + per_case
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def r1(v):
    return round(float(v), 1)


def r3(v):
    return round(float(v), 3)


def r4(v):
    return round(float(v), 4)


def _mhz(summary):
    return None if summary is None else int(summary["sm_mhz"])


def secondary_measurements(mxq, dev, stream, hbm, bf16_peak, Ws, clocks):
    """Every other measured configuration, as compact entries: name ``n``,
    time ``us``, TFLOP/s ``TF`` and/or GB/s ``GBs``, the binding roofline
    ``bound`` and the fraction of it reached ``frac``, and the median SM
    clock ``mhz`` while it ran.  The list ends with the workload
    configurations, so that they close the JSON line."""
    import torch

    out = []
    iters = 40

    def entry(name, t, nbytes, flops, m0, extra=None):
        t_mem = nbytes / (hbm * 1e9)
        t_fl = flops / (bf16_peak * 1e12) if flops else 0.0
        bound = "hbm" if t_mem >= t_fl else "tensor"
        e = {"n": name, "us": r3(t * 1e6), "GBs": r1(nbytes / t / 1e9)}
        if flops:
            e["TF"] = r1(flops / t / 1e12)
        e["bound"] = bound
        e["frac"] = r4(max(t_mem, t_fl) / t)
        e["mhz"] = _mhz(clocks.summary(m0))
        if extra:
            e.update(extra)
        return e

    def dense_entry(name, M, K, N, bits, W, copies, group=64):
        d = DenseInputs(W, M, K, N, bits, dev, copies=copies, group=group)
        if M == 1:
            fn = lambda i: mxq.qmv(d.x[0], *d.copies[i % copies], bits, out=d.y[0],  # noqa: E731
                                   group_size=group)
        else:
            fn = lambda i: mxq.qmm(d.x, *d.copies[i % copies], bits, out=d.y,  # noqa: E731
                                   group_size=group)
        for i in range(5):
            fn(i)
        m0 = clocks.mark()
        t, _ = time_launches(fn, iters, stream)
        del d
        return entry("%s M=%d K=%d N=%d b%d g%d" % (name, M, K, N, bits, group), t,
                     qmm_bytes(M, K, N, bits, group), 2.0 * M * K * N if M > 1 else 0.0, m0)

    W_big = Ws.get((5120, 17408))
    if W_big is None:
        W_big = synth.dense_weights(17408, 5120, seed=0)
    W_sq = synth.dense_weights(5120, 5120, seed=0)

    # ---- other widths and group sizes on the decode and prefill shapes
    for bits in (2, 3, 6):
        out.append(dense_entry("qmv", 1, 5120, 17408, bits, W_big, copies=6))
        out.append(dense_entry("qmm", 600, 5120, 17408, bits, W_big, copies=3))
    for group in (32, 128):
        out.append(dense_entry("qmv", 1, 5120, 17408, 4, W_big, copies=6, group=group))
        out.append(dense_entry("qmm", 600, 5120, 17408, 4, W_big, copies=3, group=group))

    # ---- the decode GEMV for the [K, N] operand layout (codes and groups along n)
    for (K, N) in ((5120, 17408), (17408, 5120)):
        Wkn = synth.dense_weights(K, N, seed=0)
        qkn = synth.quantize(Wkn, 4)
        kn_copies = [(dev_codes(qkn.w, dev), dev_bf16(qkn.scales, dev), dev_bf16(qkn.biases, dev))]
        kn_copies += [tuple(t.clone() for t in kn_copies[0]) for _ in range(5)]
        xkn = dev_bf16(synth.activations(1, K, seed=1), dev)[0]
        ykn = torch.empty((N,), dtype=torch.bfloat16, device=dev)
        fnk = lambda i: mxq.qmv_kn(xkn, *kn_copies[i % 6], 4, out=ykn)  # noqa: E731
        for i in range(5):
            fnk(i)
        m0 = clocks.mark()
        tk, _ = time_launches(fnk, iters, stream)
        out.append(entry("qmv_kn K=%d N=%d b4 g64" % (K, N), tk, qmv_bytes(K, N, 4), 0.0, m0))
        del kn_copies, Wkn, qkn
    torch.cuda.empty_cache()

    # ---- the [K, N]-layout tensor-core GEMMs: the prefill shape and both
    # expert shapes of the sorted-MoE workload (weights quantised along n
    # by the library's encoder: a [K, N] matrix quantised row by row)
    for bits in (4, 8):
        K, N, M = 5120, 17408, 600
        Wd = torch.randn((K, N), device=dev) * 0.02
        knc = [mxq.quantize(Wd, bits)]
        knc += [tuple(t.clone() for t in knc[0]) for _ in range(2)]
        del Wd
        xk = dev_bf16(synth.activations(M, K, seed=1), dev)
        yk = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fnk = lambda i: mxq.qmm_kn(xk, *knc[i % 3], bits, out=yk)  # noqa: E731
        for i in range(5):
            fnk(i)
        m0 = clocks.mark()
        tk, _ = time_launches(fnk, iters, stream)
        out.append(entry("qmm_kn M=%d K=%d N=%d b%d g64" % (M, K, N, bits), tk,
                         qmm_bytes(M, K, N, bits), 2.0 * M * K * N, m0))
        del knc, xk, yk
    for K, N, ident in ((2816, 704, False), (704, 2816, True)):
        E, T, top_k, bits = 128, 573, 8, 4
        ids, src = synth.routing(T, E, top_k, seed=2)
        B = ids.shape[0]
        We = torch.randn((E * K, N), device=dev) * 0.02
        c0, s0, b0 = mxq.quantize(We, bits)
        del We
        knc = [(c0.view(E, K, -1), s0.view(E, K, -1), b0.view(E, K, -1))]
        knc.append(tuple(t.clone() for t in knc[0]))
        Tx = B if ident else T
        xg = dev_bf16(synth.activations(Tx, K, seed=1), dev)
        ids_d = torch.from_numpy(ids).to(dev)
        src_d = None if ident else torch.from_numpy(src).to(dev)
        yg = torch.empty((B, N), dtype=torch.bfloat16, device=dev)
        wsk = torch.empty((mxq.gather_workspace_bytes(B, E, K, N),), dtype=torch.uint8, device=dev)
        fng = lambda i: mxq.gather_qmm_kn(xg, *knc[i % 2], ids_d, src_d, bits,  # noqa: E731
                                          out=yg, workspace=wsk)
        for i in range(5):
            fng(i)
        m0 = clocks.mark()
        tg, _ = time_launches(fng, iters, stream)
        nbg = E * (K * N * bits // 8 + K * (N // 64) * 4) + Tx * K * 2 + B * N * 2
        out.append(entry("gather_qmm_kn E=128 top8 T=573 B=%d K=%d N=%d b4 g64" % (B, K, N), tg,
                         nbg, 2.0 * B * K * N, m0))
        del knc, c0, s0, b0, xg, yg, wsk
    torch.cuda.empty_cache()

    # ---- the encoder on the prefill weight shape (float32 in, 4-bit codes out)
    N_q, K_q = 17408, 5120
    Wq = [torch.randn((N_q, K_q), device=dev) * 0.02 for _ in range(2)]
    cq = torch.empty((N_q, K_q // 8), dtype=torch.int32, device=dev)
    sq = torch.empty((N_q, K_q // 64), dtype=torch.bfloat16, device=dev)
    bq = torch.empty((N_q, K_q // 64), dtype=torch.bfloat16, device=dev)
    fnq = lambda i: mxq.quantize(Wq[i % 2], 4, codes=cq, scales=sq, biases=bq)  # noqa: E731
    for i in range(3):
        fnq(i)
    m0 = clocks.mark()
    tq, _ = time_launches(fnq, iters, stream)
    nbq = N_q * K_q * 4 + N_q * K_q // 2 + N_q * (K_q // 64) * 4
    out.append(entry("quantize f32 [17408,5120] -> b4 g64", tq, nbq, 0.0, m0))
    del Wq, cq, sq, bq
    torch.cuda.empty_cache()

    # ---- sorted MoE: experts of both shapes, the decode-sized calls first
    workload = []
    for K, N, ident in ((2816, 704, False), (704, 2816, True)):
        E, T, top_k, bits = 128, 573, 8, 4
        ids, src = synth.routing(T, E, top_k, seed=2)
        B = ids.shape[0]
        wl, sl, bl = [], [], []
        for e in range(E):
            q = synth.quantize(synth.dense_weights(N, K, seed=e), bits)
            wl.append(q.w)
            sl.append(q.scales)
            bl.append(q.biases)
        w = dev_codes(np.stack(wl), dev)
        s = dev_bf16(np.stack(sl), dev)
        b = dev_bf16(np.stack(bl), dev)
        copies = [(w, s, b), (w.clone(), s.clone(), b.clone())]
        # the up projection's weights for the gate/up pair: two more copies,
        # so that no launch finds either set in L2
        ucopies = [(w.clone(), s.clone(), b.clone()) for _ in range(2)] if not ident else None
        expert_bytes = N * K * bits // 8 + N * (K // 64) * 4
        wsz = torch.empty((mxq.gather_workspace_bytes(B, E, K, N),), dtype=torch.uint8,
                          device=dev)
        # decode-sized calls on the same experts: a few tokens x top 8
        for tokens in (4, 16, 64, 128):
            idsd, srcd = synth.routing(tokens, E, top_k, seed=3)
            Bd = idsd.shape[0]
            xd = dev_bf16(synth.activations(Bd if ident else tokens, K, seed=1), dev)
            idsd_d = torch.from_numpy(idsd).to(dev)
            srcd_d = None if ident else torch.from_numpy(srcd).to(dev)
            yd = torch.empty((Bd, N), dtype=torch.bfloat16, device=dev)
            fnd = lambda i: mxq.gather_qmm(xd, *copies[i % 2], idsd_d, srcd_d, bits,  # noqa: E731
                                           out=yd, workspace=wsz)
            for i in range(5):
                fnd(i)
            m0 = clocks.mark()
            td, _ = time_launches(fnd, iters, stream)
            used = len(set(idsd.tolist()))
            nbd = used * expert_bytes + xd.numel() * 2 + Bd * N * 2
            out.append(entry("gather decode T=%d B=%d K=%d N=%d b4" % (tokens, Bd, K, N), td, nbd,
                             0.0, m0, {"experts": used}))
            if not ident:
                # the gate/up pair on the same routing: a second expert set
                yu = torch.empty((Bd, N), dtype=torch.bfloat16, device=dev)
                fng = lambda i: mxq.gather_qmm_gateup(  # noqa: E731
                    xd, *copies[i % 2], *ucopies[i % 2], idsd_d, srcd_d, bits, out_gate=yd,
                    out_up=yu, workspace=wsz)
                for i in range(5):
                    fng(i)
                m0 = clocks.mark()
                tg, _ = time_launches(fng, iters, stream)
                nbg = 2 * used * expert_bytes + xd.numel() * 2 + 2 * Bd * N * 2
                out.append(entry("gateup decode T=%d B=%d K=%d N=%d b4" % (tokens, Bd, K, N), tg,
                                 nbg, 0.0, m0, {"experts": used}))
        Tx = B if ident else T
        x = dev_bf16(synth.activations(Tx, K, seed=1), dev)
        ids_d = torch.from_numpy(ids).to(dev)
        src_d = None if ident else torch.from_numpy(src).to(dev)
        y = torch.empty((B, N), dtype=torch.bfloat16, device=dev)
        fn = lambda i: mxq.gather_qmm(x, *copies[i % 2], ids_d, src_d, bits, out=y,  # noqa: E731
                                      workspace=wsz)
        for i in range(5):
            fn(i)
        m0 = clocks.mark()
        t, _ = time_launches(fn, iters, stream)
        nbytes = E * expert_bytes + Tx * K * 2 + B * N * 2
        workload.append(entry("gather_qmm E=128 top8 T=573 B=%d K=%d N=%d b4 g64" % (B, K, N), t,
                           nbytes, 2.0 * B * K * N, m0, {"tok_s": int(T / t)}))
        del w, s, b, copies, ucopies, x, y
        torch.cuda.empty_cache()

    # ---- the workload configurations: M sweep at K=N=5120, the 4/8-bit pair,
    # then the prefill GEMM
    sweep = [dense_entry("qmm", M, 5120, 5120, 4, W_sq, copies=6) for M in (1, 8, 32, 128, 600)]
    pair = [dense_entry("pair qmv", 1, 5120, 5120, 8, W_sq, copies=6),
            dense_entry("pair qmm", 128, 5120, 5120, 8, W_sq, copies=6)]
    prefill = dense_entry("qmm prefill", 600, 5120, 17408, 4, W_big, copies=3)
    prefill["tok_s"] = int(600 / (prefill["us"] * 1e-6))
    return out + workload + sweep + pair + [prefill]



# ------------------------------------------------------------------ CPU side


def cpu_baseline(seconds):
    """The f64 checker on the host cores: qmv K=5120 N=17408 4-bit, whole
    output, repeated for about ``seconds``."""
    import oracle

    K, N, bits = 5120, 17408, 4
    qw = synth.quantize(synth.dense_weights(N, K, seed=0), bits)
    x = synth.activations(1, K, seed=1)
    oracle.qmv(x[0], qw.w, qw.scales, qw.biases, K, N, bits)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.qmv(x[0], qw.w, qw.scales, qw.biases, K, N, bits)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(qmv_bytes(K, N, bits) / dt / 1e9, 3), "unit": "GB/s",
            "cores": oracle.threads(), "kind": "oracle",
            "sample": "f64 qmv K=5120 N=17408 4-bit, whole output, %d repetitions" % reps}


def run_reference(args):
    """The f64 checker as the reference arm, on the host cores.  A step is
    the decode step (all four cases) over a sample of each case's output
    rows, sized so that warm-up plus timed steps take about
    ``--reference-seconds``; the sample rotates through the rows from step
    to step.  Under torchrun only rank 0 runs; the other ranks exit at once."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    cases = []
    Ws = {}
    for K, N, bits in DECODE_CASES:
        if (K, N) not in Ws:
            Ws[(K, N)] = synth.dense_weights(N, K, seed=0)
        qw = synth.quantize(Ws[(K, N)], bits)
        cases.append((K, N, bits, qw, synth.activations(1, K, seed=1)))

    def run_rows(frac, step_index):
        """All four cases over ceil(frac * N) rows each; returns the bytes."""
        nbytes = 0
        for K, N, bits, qw, x in cases:
            rows = max(1, min(N, int(np.ceil(frac * N))))
            r0 = (step_index * rows) % N
            r1 = min(N, r0 + rows)
            oracle.qmv(x[0], qw.w[r0:r1], qw.scales[r0:r1], qw.biases[r0:r1], K, r1 - r0, bits)
            nbytes += (r1 - r0) * (K * bits // 8 + (K // 64) * 4 + 2) + K * 2
        return nbytes

    # size the sample: one full step timed once, then the fraction of rows
    # that fits the time budget
    t0 = time.perf_counter()
    run_rows(1.0, 0)
    t_full = time.perf_counter() - t0
    per_step = args.reference_seconds / (args.steps + args.warmup)
    frac = min(1.0, per_step / t_full)
    for i in range(args.warmup):
        run_rows(frac, i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        nbytes += run_rows(frac, args.warmup + i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    rows = [max(1, min(N, int(np.ceil(frac * N)))) for K, N, bits, _, _ in cases]
    sample = ("f64 checker, all four decode cases per step, %s output rows of N=%s per step "
              "(%.4g of each matrix, rotating)" % (rows, [c[1] for c in cases], frac))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": CONFIG,
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """A few plain launches of one workload, for ncu (no graphs, no timing)."""
    import torch

    import affine_bit_matmul_gb300 as mxq
    from affine_bit_matmul_gb300 import build as _build

    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = args.profile
    launches = args.profile_launches
    if name == "decode":
        for K, N, bits in DECODE_CASES:
            d = DenseInputs(synth.dense_weights(N, K, seed=0), 1, K, N, bits, dev, copies=2)
            for i in range(launches):
                mxq.qmv(d.x[0], *d.copies[i % 2], bits, out=d.y[0])
            torch.cuda.synchronize()
            del d
    elif name.startswith("qmv"):
        K, N, bits = {"qmv4": (5120, 17408, 4), "qmv8": (5120, 17408, 8),
                      "qmv4t": (17408, 5120, 4), "qmv8t": (17408, 5120, 8)}[name]
        d = DenseInputs(synth.dense_weights(N, K, seed=0), 1, K, N, bits, dev, copies=2)
        for i in range(launches):
            mxq.qmv(d.x[0], *d.copies[i % 2], bits, out=d.y[0])
    elif name == "qmm_kn":
        # the [K, N]-layout prefill GEMM: weights quantised along n by the
        # library's encoder
        M, K, N, bits = 600, 5120, 17408, 4
        c = mxq.quantize(torch.randn((K, N), device=dev) * 0.02, bits)
        x = dev_bf16(synth.activations(M, K, seed=1), dev)
        for i in range(launches):
            mxq.qmm_kn(x, *c, bits)
    elif name.startswith("qmm"):
        M, K, N, bits = {"qmm": (600, 5120, 17408, 4), "qmm600": (600, 5120, 5120, 4),
                         "qmm128": (128, 5120, 5120, 4), "qmm8": (8, 5120, 5120, 4),
                         "qmm2": (2, 5120, 5120, 4), "qmm32": (32, 5120, 5120, 4)}[name]
        d = DenseInputs(synth.dense_weights(N, K, seed=0), M, K, N, bits, dev, copies=2)
        for i in range(launches):
            mxq.qmm(d.x, *d.copies[i % 2], bits, out=d.y)
    else:
        K, N, ident = {"gather_up": (2816, 704, False), "gather_down": (704, 2816, True),
                       "gather_up_t4": (2816, 704, False),
                       "gather_down_t4": (704, 2816, True)}[name]
        E, T, top_k, bits = 128, 573, 8, 4
        if name.endswith("_t4"):
            T = 4  # a decode step of 4 tokens: 32 routed rows
        ids, src = synth.routing(T, E, top_k, seed=2)
        B = ids.shape[0]
        rng = np.random.default_rng(0)
        # timing-only inputs: random codes, small scales
        w = torch.from_numpy(rng.integers(0, 2 ** 31, size=(E, N, K // 8), dtype=np.int32)).to(dev)
        s = torch.full((E, N, K // 64), 0.001, dtype=torch.bfloat16, device=dev)
        b = torch.full((E, N, K // 64), -0.01, dtype=torch.bfloat16, device=dev)
        Tx = B if ident else T
        x = dev_bf16(synth.activations(Tx, K, seed=1), dev)
        ids_d = torch.from_numpy(ids).to(dev)
        src_d = None if ident else torch.from_numpy(src).to(dev)
        for i in range(launches):
            mxq.gather_qmm(x, w, s, b, ids_d, src_d, bits)
    torch.cuda.synchronize()
    print("profile run done: %s x%d" % (name, launches))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None,
                    help="plain launches of one workload for ncu: decode qmv4 qmv8 qmv4t qmv8t qmm "
                         "qmm600 qmm128 qmm8 qmm2 qmm32 gather_up gather_down gather_up_t4 "
                         "gather_down_t4")
    ap.add_argument("--profile-launches", type=int, default=4)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mxq", "reference"], default="mxq")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="time budget of the reference arm (warm-up + timed steps)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="issue every launch directly instead of through CUDA graphs")
    args = ap.parse_args()
    if args.no_graphs:
        global USE_GRAPHS
        USE_GRAPHS = False
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_mxq(args)


if __name__ == "__main__":
    main()
