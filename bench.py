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
    """nvidia-smi sampling of SM clocks and throttle reasons."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
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
        rows = [l.strip().split(",") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sms.append(float(r[1]))
                maxes.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


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


def time_launches(fn, iters, stream, reps=5):
    """Median per-launch device time of fn over graphs of ``iters`` launches
    (CUDA events on the launching stream around each graph replay)."""
    import torch

    g = capture(fn, iters)
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
    for i in range(args.warmup):
        graphs[i % 2].replay()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
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
    clk = clocks.stop()
    local_elapsed = t0.elapsed_time(t1) * 1e-3
    elapsed = max_over_ranks(local_elapsed, world)
    value = step_bytes * args.steps * world / elapsed / 1e9
    # the timed region holds nothing but qmv launches (four per step): the
    # kernel's algorithmic bytes per launch over its mean launch duration
    # there is this rank's step bytes over its time per step
    achieved = step_bytes * args.steps / local_elapsed / 1e9

    # per-case device time, each case alone (graphs of 20 launches): the
    # breakdown of the step, not the roofline figure
    per_case = []
    for c in cases:
        t, _ = time_launches(
            lambda i, c=c: mxq.qmv(c.x[0], *c.copies[i % 2], c.bits, out=c.y[0]), 20, stream)
        nb = qmv_bytes(c.K, c.N, c.bits)
        per_case.append({"K": c.K, "N": c.N, "bits": c.bits, "us": t * 1e6, "GB_s": nb / t / 1e9,
                         "frac_hbm": nb / t / 1e9 / hbm})

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
        secondary = secondary_measurements(mxq, dev, stream, hbm, bf16_peak, Ws)

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
        "config": {"workload": WORKLOAD, "M": 1, "group_size": 64,
                   "l2": "inputs larger than L2: each case alternates two input copies "
                         "(580 MB working set vs 129 MB L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "qmv_stream_kernel (4- and 8-bit)",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic_per_launch(),
                     "algorithmic_bytes_per_launch": step_bytes // len(cases),
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"},
        "per_case": per_case,
        "gpu_launches": len(cases) * args.steps,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "public API qmv with inputs copied from pinned host memory every step"},
        "clocks": clk,
        "secondary": secondary,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def secondary_measurements(mxq, dev, stream, hbm, bf16_peak, Ws):
    """Prefill GEMM, M sweep, the 4/8-bit pair, other bit widths and group sizes,
    the [K, N] layout GEMV, the encoder and the sorted-MoE gather."""
    import torch

    out = []
    iters = 40

    def dense_entry(name, M, K, N, bits, W, copies, group=64):
        d = DenseInputs(W, M, K, N, bits, dev, copies=copies, group=group)
        if M == 1:
            fn = lambda i: mxq.qmv(d.x[0], *d.copies[i % copies], bits, out=d.y[0],  # noqa: E731
                                   group_size=group)
            kern = "qmv_stream_kernel"
        else:
            fn = lambda i: mxq.qmm(d.x, *d.copies[i % copies], bits, out=d.y,  # noqa: E731
                                   group_size=group)
            kern = "qmm_tc_kernel or qmm_persistent_kernel"
        for i in range(5):
            fn(i)
        t, _ = time_launches(fn, iters, stream)
        flops = 2.0 * M * K * N
        nbytes = qmm_bytes(M, K, N, bits, group)
        t_star = max(nbytes / (hbm * 1e9), flops / (bf16_peak * 1e12))
        bound = "hbm" if nbytes / (hbm * 1e9) >= flops / (bf16_peak * 1e12) else "tensor"
        del d
        return {"name": name, "kernel": kern, "M": M, "K": K, "N": N, "bits": bits,
                "group": group, "us": t * 1e6, "TFLOPS": flops / t / 1e12, "GB_s": nbytes / t / 1e9,
                "frac_tensor": flops / t / 1e12 / bf16_peak, "frac_hbm": nbytes / t / 1e9 / hbm,
                "bound": bound, "frac_roofline": t_star / t, "tokens_per_s": M / t}

    W_big = Ws.get((5120, 17408)) if Ws.get((5120, 17408)) is not None else synth.dense_weights(
        17408, 5120, seed=0)
    out.append(dense_entry("qmm prefill", 600, 5120, 17408, 4, W_big, copies=3))
    W_sq = synth.dense_weights(5120, 5120, seed=0)
    for M in (1, 8, 32, 128, 600):
        out.append(dense_entry("qmm sweep", M, 5120, 5120, 4, W_sq, copies=6))
    # controlled pair: same W, 8-bit (4-bit rows are in the sweep above)
    out.append(dense_entry("pair qmv 8-bit", 1, 5120, 5120, 8, W_sq, copies=6))
    out.append(dense_entry("pair qmv 4-bit", 1, 5120, 5120, 4, W_sq, copies=6))
    out.append(dense_entry("pair qmm 8-bit", 128, 5120, 5120, 8, W_sq, copies=6))
    # 2-, 3- and 6-bit codes and group sizes 32 and 128 on the decode and
    # prefill shapes (same weights)
    for bits in (2, 3, 6):
        out.append(dense_entry("%d-bit qmv" % bits, 1, 5120, 17408, bits, W_big, copies=6))
        out.append(dense_entry("%d-bit qmm prefill" % bits, 600, 5120, 17408, bits, W_big,
                               copies=3))
    for group in (32, 128):
        out.append(dense_entry("group qmv", 1, 5120, 17408, 4, W_big, copies=6, group=group))
        out.append(dense_entry("group qmm prefill", 600, 5120, 17408, 4, W_big, copies=3,
                               group=group))

    # the decode GEMV for the [K, N] operand layout (codes and groups along n)
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
        tk, _ = time_launches(fnk, iters, stream)
        nbk = qmv_bytes(K, N, 4)
        out.append({"name": "qmv [K, N] layout", "kernel": "qmv_kn_kernel", "M": 1, "K": K,
                    "N": N, "bits": 4, "group": 64, "us": tk * 1e6,
                    "TFLOPS": 2.0 * K * N / tk / 1e12, "GB_s": nbk / tk / 1e9,
                    "frac_hbm": nbk / tk / 1e9 / hbm, "bound": "hbm",
                    "frac_roofline": nbk / tk / 1e9 / hbm, "tokens_per_s": 1 / tk})
        del kn_copies, Wkn, qkn
    torch.cuda.empty_cache()

    # the encoder on the prefill weight shape (float32 in, 4-bit codes out)
    N_q, K_q = 17408, 5120
    Wq = [torch.randn((N_q, K_q), device=dev) * 0.02 for _ in range(2)]
    cq = torch.empty((N_q, K_q // 8), dtype=torch.int32, device=dev)
    sq = torch.empty((N_q, K_q // 64), dtype=torch.bfloat16, device=dev)
    bq = torch.empty((N_q, K_q // 64), dtype=torch.bfloat16, device=dev)
    fnq = lambda i: mxq.quantize(Wq[i % 2], 4, codes=cq, scales=sq, biases=bq)  # noqa: E731
    for i in range(3):
        fnq(i)
    tq, _ = time_launches(fnq, iters, stream)
    nbq = N_q * K_q * 4 + N_q * K_q // 2 + N_q * (K_q // 64) * 4
    out.append({"name": "quantize", "kernel": "quantize_kernel", "K": K_q, "N": N_q, "bits": 4,
                "us": tq * 1e6, "TFLOPS": 0.0, "GB_s": nbq / tq / 1e9,
                "frac_hbm": nbq / tq / 1e9 / hbm, "bound": "hbm",
                "frac_roofline": nbq / tq / 1e9 / hbm, "tokens_per_s": 0.0})
    del Wq, cq, sq, bq
    torch.cuda.empty_cache()

    # sorted MoE gather, both expert shapes
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
        Tx = B if ident else T
        x = dev_bf16(synth.activations(Tx, K, seed=1), dev)
        ids_d = torch.from_numpy(ids).to(dev)
        src_d = None if ident else torch.from_numpy(src).to(dev)
        y = torch.empty((B, N), dtype=torch.bfloat16, device=dev)
        wsz = torch.empty((mxq.gather_workspace_bytes(B, E, K if src_d is not None else 0, N),), dtype=torch.uint8, device=dev)
        fn = lambda i: mxq.gather_qmm(x, *copies[i % 2], ids_d, src_d, bits, out=y,  # noqa: E731
                                      workspace=wsz)
        for i in range(5):
            fn(i)
        t, _ = time_launches(fn, iters, stream)
        flops = 2.0 * B * K * N
        nbytes = E * (N * K * bits // 8 + N * (K // 64) * 4) + Tx * K * 2 + B * N * 2
        t_star = max(nbytes / (hbm * 1e9), flops / (bf16_peak * 1e12))
        out.append({"name": "gather_qmm", "kernel": "gather_prepass + gather_rows + qmm_persistent_kernel",
                    "E": E, "top_k": top_k, "tokens": T, "B": B, "K": K, "N": N, "bits": bits,
                    "us": t * 1e6, "TFLOPS": flops / t / 1e12, "GB_s": nbytes / t / 1e9,
                    "frac_tensor": flops / t / 1e12 / bf16_peak, "frac_hbm": nbytes / t / 1e9 / hbm,
                    "bound": "hbm", "frac_roofline": t_star / t, "tokens_per_s": T / t})
        # decode-sized call on the same experts: 4 tokens x top 8 = 32 rows
        ids4, src4 = synth.routing(4, E, top_k, seed=3)
        B4 = ids4.shape[0]
        x4 = dev_bf16(synth.activations(B4 if ident else 4, K, seed=1), dev)
        ids4_d = torch.from_numpy(ids4).to(dev)
        src4_d = None if ident else torch.from_numpy(src4).to(dev)
        y4 = torch.empty((B4, N), dtype=torch.bfloat16, device=dev)
        fn4 = lambda i: mxq.gather_qmm(x4, *copies[i % 2], ids4_d, src4_d, bits, out=y4,  # noqa: E731
                                       workspace=wsz)
        for i in range(5):
            fn4(i)
        t4, _ = time_launches(fn4, iters, stream)
        used = len(set(ids4.tolist()))
        nb4 = used * (N * K * bits // 8 + N * (K // 64) * 4) + x4.numel() * 2 + B4 * N * 2
        out.append({"name": "gather_qmm decode", "kernel": "gather_qmv_kernel",
                    "E": E, "top_k": top_k, "tokens": 4, "B": B4, "experts_used": used, "K": K,
                    "N": N, "bits": bits, "us": t4 * 1e6, "TFLOPS": 2.0 * B4 * K * N / t4 / 1e12,
                    "GB_s": nb4 / t4 / 1e9, "frac_hbm": nb4 / t4 / 1e9 / hbm, "bound": "hbm",
                    "frac_roofline": nb4 / t4 / 1e9 / hbm, "tokens_per_s": 4 / t4})
        del w, s, b, copies, x, y
        torch.cuda.empty_cache()
    return out


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
        "config": {"workload": WORKLOAD, "M": 1, "group_size": 64},
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
    elif name.startswith("qmm"):
        M, K, N, bits = {"qmm": (600, 5120, 17408, 4), "qmm600": (600, 5120, 5120, 4),
                         "qmm128": (128, 5120, 5120, 4), "qmm8": (8, 5120, 5120, 4),
                         "qmm32": (32, 5120, 5120, 4)}[name]
        d = DenseInputs(synth.dense_weights(N, K, seed=0), M, K, N, bits, dev, copies=2)
        for i in range(launches):
            mxq.qmm(d.x, *d.copies[i % 2], bits, out=d.y)
    else:
        K, N, ident = {"gather_up": (2816, 704, False), "gather_down": (704, 2816, True)}[name]
        E, T, top_k, bits = 128, 573, 8, 4
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
                         "qmm600 qmm128 qmm8 qmm32 gather_up gather_down")
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
