"""Benchmark of the W4A16 decode hot path on GB300 (one JSON line on stdout).

Workload (one "step"): the W4A16 decode GEMMs of Llama-7B-like layers -- M in
{1, 16} tokens x (N, K) in {(4096, 4096), (11008, 4096), (4096, 11008),
(12288, 4096)}, group size 128, fp16 activations ~ N(0, 1), codes uniform over
0..15, fp16 scales ~ U[0.005, 0.02] -- eight GEMMs through libwq.so.

Metric: HBM GB/s over the algorithmic bytes (packed weight + scales + A + out),
as a fraction of the measured copy bandwidth.  Extras on the same line: per-GEMM
microseconds, the M = 4096 prefill GEMMs in TFLOP/s against the measured dense
bf16/fp16 tensor peak, an end-to-end figure through the public API with pinned
host buffers, and the float64 CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference that exists for this
method) on a bounded sample of the same workload.  Under torchrun every rank
runs an independent replica (the decode GEMMs do not shard); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM µs + HBM GB/s (M<=16) / TFLOP/s (M=4096), % of roofline"
DECODE_SHAPES = [(4096, 4096), (11008, 4096), (4096, 11008), (12288, 4096)]
DECODE_M = (1, 16)
G = 128
ROTATING_SETS = 3
WORKLOAD = ("W4A16 decode, Llama-7B-like layers: M in {1,16} x (N,K) in {(4096,4096),(11008,4096),"
            "(4096,11008),(12288,4096)}, group_size 128, fp16 A ~N(0,1), q uniform 0..15, "
            "scales fp16 ~U[0.005,0.02]; one step = the 8 GEMMs")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algo_bytes(M, N, K, G_):
    return N * K // 2 + (K // G_) * N * 2 + M * K * 2 + M * N * 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The sources the decode kernel is compiled from (its own header, the helpers and PTX
# wrappers it includes, the shared declarations and the instantiating unit).
DECODE_KERNEL_SOURCES = ("wq_gemm_mma.cuh", "wq_common.cuh", "sm103_ptx.cuh", "wq_internal.h", "wq_gemm_int4.cu")


def kernel_source_hash():
    h = hashlib.sha256()
    for name in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "weight_only_quantized_tma_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(plan_of=None):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on
    the current kernel sources and the captured shape still gets the recorded launch
    (grid and K slices); else None."""
    path = os.path.join(ROOT, "profiles", "wq_gemm_w4a16_decode_ncu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        if plan_of is not None:
            M, N, K, Gc = (int(x) for x in vals["captured_shape"].split(","))
            plan = plan_of(M, N, K, Gc)
            if plan["grid"] != int(vals["captured_grid"]) or plan["splits"] != int(vals["captured_splits"]):
                return None
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"wq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # nvidia-smi takes a moment to print its first line: wait for it (bounded) so
        # the sampler is live when the timed region starts
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 5.0:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                break
            time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_decode(step_fraction_cols, min_seconds, seed_base=1000):
    """Time the float64 oracle on the decode workload: every GEMM of the step, on a
    column (weight-row) sample of the given fraction.  Returns (GB/s, seconds, cores, sample)."""
    import oracle
    from weight_only_quantized_tma_gb300 import synth
    problems = []
    for mi, M in enumerate(DECODE_M):
        for si, (N, K) in enumerate(DECODE_SHAPES):
            seed = synth.seed_for(1, mi * len(DECODE_SHAPES) + si)
            A = synth.activations(M, K, "f16", seed)
            w = synth.int4_weights(N, K, G, seed + 1)
            ncols = max(1, int(round(N * step_fraction_cols)))
            cols = np.linspace(0, N - 1, ncols).astype(np.int64)
            problems.append((M, N, K, A, w, cols))
    oracle.build()
    byts, elapsed, reps = 0.0, 0.0, 0
    while True:
        t0 = time.perf_counter()
        for (M, N, K, A, w, cols) in problems:
            oracle.gemm_w4a16(A, False, w.w, w.s, M, N, K, G, cols=cols)
            frac = len(cols) / N
            byts += algo_bytes(M, N, K, G) * frac
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed >= min_seconds:
            break
    sample = (f"{reps} pass(es) over all 8 decode GEMMs, {step_fraction_cols:.4g} of the weight rows "
              f"(output columns) of each, all M tokens")
    return byts / elapsed / 1e9, elapsed, oracle.num_threads(), sample


def max_over_ranks(x, world, device="cpu"):
    """The largest value over all ranks (the slowest rank's time); x itself on one rank."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    if rank != 0:
        return
    # each step: the oracle on 1/64 of the output columns of every decode GEMM
    frac = 1.0 / 64
    import oracle
    from weight_only_quantized_tma_gb300 import synth
    problems = []
    for mi, M in enumerate(DECODE_M):
        for si, (N, K) in enumerate(DECODE_SHAPES):
            seed = synth.seed_for(1, mi * len(DECODE_SHAPES) + si)
            cols = np.linspace(0, N - 1, max(1, int(N * frac))).astype(np.int64)
            problems.append((M, N, K, synth.activations(M, K, "f16", seed), synth.int4_weights(N, K, G, seed + 1),
                             cols))
    oracle.build()

    def step():
        b = 0.0
        for (M, N, K, A, w, cols) in problems:
            oracle.gemm_w4a16(A, False, w.w, w.s, M, N, K, G, cols=cols)
            b += algo_bytes(M, N, K, G) * len(cols) / N
        return b

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    byts = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = byts / dt / 1e9
    sample = f"each step: all 8 decode GEMMs on {frac:.4g} of their output columns (weight rows), all M tokens"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "impl": "float64 CPU oracle (oracle/oracle.c)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import weight_only_quantized_tma_gb300 as wq
    from weight_only_quantized_tma_gb300 import build as wq_build
    from weight_only_quantized_tma_gb300 import synth

    wq_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peaks, peaks_src = load_peaks()

    # ---------------- inputs (resident in HBM before timing); 3 rotating weight sets > L2
    gemms = []   # per set: list of (M, N, K, A, wk, sk, out)
    with torch.cuda.stream(stream):
        for r in range(ROTATING_SETS):
            sets = []
            for mi, M in enumerate(DECODE_M):
                for si, (N, K) in enumerate(DECODE_SHAPES):
                    seed = synth.seed_for(1, mi * len(DECODE_SHAPES) + si) + 100 * r
                    A = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.float16)).to(dev)
                    w = synth.int4_weights(N, K, G, seed + 1)
                    wk, sk = wq.wq_pack_int4(torch.from_numpy(w.w).to(dev),
                                             torch.from_numpy(w.s.view(np.float16)).to(dev), N, K, G)
                    out = torch.empty((M, N), dtype=torch.float16, device=dev)
                    sets.append((M, N, K, A, wk, sk, out))
            gemms.append(sets)
        max_ws = max(wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)["ws_bytes"]
                     for (M, N, K, *_r) in gemms[0])
        ws = torch.zeros(max(max_ws, 16384), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    step_bytes = sum(algo_bytes(M, N, K, G) for (M, N, K, *_r) in gemms[0])
    launches_per_step = len(gemms[0])

    def launch_set(sets):
        for (M, N, K, A, wk, sk, out) in sets:
            wq.wq_gemm_w4a16(A, wk, sk, N, K, G, out=out, ws=ws)

    # ---------------- CUDA graphs, one per weight set
    graphs = []
    with torch.cuda.stream(stream):
        launch_set(gemms[0])   # warm the plan / function attributes before capture
        torch.cuda.synchronize(dev)
        for r in range(ROTATING_SETS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                launch_set(gemms[r])
            graphs.append(g)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---------------- warmup + timed region (graph replays, rotating weight sets)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % ROTATING_SETS].replay()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(args.steps):
                graphs[i % ROTATING_SETS].replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    step_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    # whole job: every rank (an independent replica) streams step_bytes per step
    value = step_bytes * world / (step_ms * 1e-3) / 1e9

    # ---------------- per-GEMM times inside a CUDA graph: for each decode shape, one graph of
    # back-to-back launches over rotating weight sets larger than L2 (the step's own
    # conditions: programmatic dependent launch, no host gaps), replayed 100 times
    L2_BYTES = 129e6
    per_gemm = []
    tot_bytes, tot_us = 0.0, 0.0
    for (M, N, K, A0, wk0, sk0, out0) in gemms[0]:
        nsets = max(ROTATING_SETS, int(np.ceil(2.2 * L2_BYTES / (N * K / 2))))
        with torch.cuda.stream(stream):
            sets = [(A0, wk0, sk0, out0)] + [
                (torch.randn((M, K), device=dev).to(torch.float16),
                 torch.randint(0, 256, wk0.shape, dtype=torch.uint8, device=dev), sk0,
                 torch.empty((M, N), dtype=torch.float16, device=dev)) for _ in range(nsets - 1)]
            for (A, wk, sk, out) in sets:
                wq.wq_gemm_w4a16(A, wk, sk, N, K, G, out=out, ws=ws)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for (A, wk, sk, out) in sets:
                    wq.wq_gemm_w4a16(A, wk, sk, N, K, G, out=out, ws=ws)
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(100):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(b) * 1e3 / (100 * nsets)
        byts = algo_bytes(M, N, K, G)
        tot_bytes += byts
        tot_us += us
        plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)
        per_gemm.append({"M": M, "N": N, "K": K, "us": round(us, 3), "bytes": byts,
                         "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                         "frac_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                         "splits": plan["splits"], "grid": plan["grid"], "weight_sets": nsets})
        del sets, g
    # the roofline's achieved rate: algorithmic bytes of an average launch over the
    # decode kernel's average launch duration in the timed region, where it is the
    # only kernel (8 launches per step): the step's bytes over the step time on one
    # rank.  The per-shape graphs above give each GEMM's own in-graph time.
    achieved = step_bytes / (step_ms * 1e-3) / 1e9
    per_shape_rate = tot_bytes / (tot_us * 1e-6) / 1e9
    traffic = profiled_traffic(lambda M, N, K, Gc: wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, Gc))

    # ---------------- prefill extras (M = 4096), L2 flushed between runs
    prefill = []
    if not args.skip_prefill:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        for Gp in (32, 64, 128, 256):
            M = N = K = 4096
            seed = synth.seed_for(2, (32, 64, 128, 256).index(Gp))
            A = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.float16)).to(dev)
            w = synth.int4_weights(N, K, Gp, seed + 1)
            wk, sk = wq.wq_pack_int4(torch.from_numpy(w.w).to(dev), torch.from_numpy(w.s.view(np.float16)).to(dev),
                                     N, K, Gp)
            out = torch.empty((M, N), dtype=torch.float16, device=dev)
            times = []
            with torch.cuda.stream(stream):
                for it in range(3 + 10):
                    flush.fill_(it & 0xFF)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    wq.wq_gemm_w4a16(A, wk, sk, N, K, Gp, out=out)
                    b.record(stream)
                    times.append((a, b))
            torch.cuda.synchronize(dev)
            us = statistics.median([a.elapsed_time(b) * 1e3 for a, b in times[3:]])
            tflops = 2.0 * M * N * K / (us * 1e-6) / 1e12
            prefill.append({"M": M, "N": N, "K": K, "G": Gp, "us": round(us, 2), "TFLOP/s": round(tflops, 1),
                            "frac_tensor": round(tflops / peaks["bf16_tflops"], 4)})
        del flush

    # ---------------- FP8 / FP4 extras (L2 flushed between runs): the config shapes, fp16
    # and bf16 activations, the bias epilogue, and FP4 at the FP4 page's own shape
    fp8_fp4 = []
    zero_point = []
    codebook_int2 = []
    if not args.skip_prefill:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

        def time_call(fn, reps=10):
            times = []
            with torch.cuda.stream(stream):
                for it in range(3 + reps):
                    flush.fill_(it & 0xFF)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    times.append((a, b))
            torch.cuda.synchronize(dev)
            return statistics.median([a.elapsed_time(b) * 1e3 for a, b in times[3:]])

        def graph_us(calls, reps=50):
            # back-to-back calls on distinct weight copies (together larger than L2) in
            # one CUDA graph: the per-call time without host gaps or launch ramp
            with torch.cuda.stream(stream):
                for c in calls:
                    c()
                torch.cuda.synchronize(dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for c in calls:
                        c()
                for _ in range(3):
                    g.replay()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    g.replay()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) * 1e3 / (reps * len(calls))

        def graph_fields(us, byts):
            return {"us_graph": round(us, 2), "GB/s_graph": round(byts / (us * 1e-6) / 1e9, 1),
                    "frac_hbm_graph": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}

        def n_copies(wbytes):
            return max(ROTATING_SETS, int(np.ceil(2.2 * L2_BYTES / wbytes)))

        def entry(op, M, N, K, adt, us, byts, extra=None, into=None):
            d = {"op": op, "M": M, "N": N, "K": K, "A": adt, "us": round(us, 2),
                 "TFLOP/s": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1),
                 "frac_tensor": round(2.0 * M * N * K / (us * 1e-6) / 1e12 / peaks["bf16_tflops"], 4),
                 "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                 "frac_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
            d.update(extra or {})
            (fp8_fp4 if into is None else into).append(d)

        fp8_cases = [(32768, 3200, 5120, "bf16", False), (16384, 12800, 5120, "bf16", False),
                     (8192, 10240, 5120, "bf16", False), (8192, 10240, 5120, "f16", False),
                     (8192, 10240, 5120, "f16", True), (1, 10240, 5120, "bf16", False),
                     (16, 10240, 5120, "bf16", False), (32, 10240, 5120, "bf16", False),
                     (64, 10240, 5120, "bf16", False),
                     (16, 10240, 5120, "f16", True)]
        for (M, N, K, adt, with_bias) in fp8_cases:
            seed = 4000 + M
            Ax = torch.from_numpy(synth.activations(M, K, adt, seed).view(np.int16)).to(dev).view(
                torch.bfloat16 if adt == "bf16" else torch.float16)
            w8 = synth.fp8_weights(N, K, seed + 1)
            wd = torch.from_numpy(w8.w).to(dev)
            alpha = torch.tensor([w8.scale], dtype=torch.float32, device=dev)
            bias = (torch.from_numpy(synth.bias(N, adt, seed + 2).view(np.int16)).to(dev).view(Ax.dtype)
                    if with_bias else None)
            outx = torch.empty((M, N), dtype=Ax.dtype, device=dev)
            wsx = torch.zeros(wq.get_plan(wq.WQ_OP_FP8, wq.WQ_F16 if adt == "f16" else wq.WQ_BF16, M, N, K, 0)
                             ["ws_bytes"] + 16, dtype=torch.uint8, device=dev)
            us = time_call(lambda: wq.wq_gemm_w8a16_fp8(Ax, wd, alpha, bias=bias, out=outx, ws=wsx))
            byts = N * K + M * K * 2 + M * N * 2
            extra = {"bias": with_bias}
            if M <= 128:
                copies = [wd] + [wd.clone() for _ in range(n_copies(N * K) - 1)]
                extra.update(graph_fields(graph_us([
                    (lambda w=w: wq.wq_gemm_w8a16_fp8(Ax, w, alpha, bias=bias, out=outx, ws=wsx)) for w in copies]),
                    byts))
                del copies
            extra["kernel"] = ["tile", "decode", "tile_pair"][wq.get_plan(
                wq.WQ_OP_FP8, wq.WQ_F16 if adt == "f16" else wq.WQ_BF16, M, N, K, 0)["kernel"]]
            entry("fp8", M, N, K, adt, us, byts, extra)
            del Ax, wd, outx, wsx
        fp4_cases = [(1, 12800, 5120, None), (128, 12800, 5120, None), (8192, 12800, 5120, None),
                     (128, 6656, 19968, "FP4 page (#4466) quotes 43.90 us for its cute-dsl kernel at this shape, "
                                        "SM100-class GPU, SKU not stated")]
        for (M, N, K, note) in fp4_cases:
            seed = 5000 + M
            Ax = torch.from_numpy(synth.activations(M, K, "bf16", seed).view(np.int16)).to(dev).view(torch.bfloat16)
            w4 = synth.fp4_weights(N, K, seed + 1)
            wd = torch.from_numpy(w4.w).to(dev)
            sfk = wq.wq_pack_fp4_sf(torch.from_numpy(w4.sf).to(dev), N, K)
            alpha = torch.tensor([w4.alpha], dtype=torch.float32, device=dev)
            outx = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsx = torch.zeros(wq.get_plan(wq.WQ_OP_FP4, wq.WQ_BF16, M, N, K, 0)["ws_bytes"] + 16,
                             dtype=torch.uint8, device=dev)
            us = time_call(lambda: wq.wq_gemm_bf16_fp4(Ax, wd, sfk, alpha, out=outx, ws=wsx))
            byts = N * K // 2 + N * K // 16 + M * K * 2 + M * N * 2
            extra = {"context": note} if note else {}
            extra["kernel"] = ["tile", "decode", "tile_pair"][wq.get_plan(wq.WQ_OP_FP4, wq.WQ_BF16, M, N, K, 0)["kernel"]]
            if M <= 128:
                copies = [(wd, sfk)] + [(wd.clone(), sfk.clone()) for _ in range(n_copies(N * K // 2) - 1)]
                extra.update(graph_fields(graph_us([
                    (lambda w=w, f=f: wq.wq_gemm_bf16_fp4(Ax, w, f, alpha, out=outx, ws=wsx)) for (w, f) in copies]),
                    byts))
                del copies
            entry("fp4", M, N, K, "bf16", us, byts, extra)
            del Ax, wd, outx, wsx
        # zero-point INT4 beside the symmetric format at the same shapes (both on the
        # register decode kernel at M <= 16, the tile kernels above)
        for (M, N, K, Gz) in [(16, 4096, 4096, 128), (128, 4096, 4096, 128), (4096, 4096, 4096, 128),
                              (8192, 8192, 8192, 128)]:
            seed = 6000 + M
            Ax = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.int16)).to(dev).view(torch.float16)
            wz = synth.int4_weights(N, K, Gz, seed + 1)
            wkz, skz = wq.wq_pack_int4(torch.from_numpy(wz.w).to(dev),
                                       torch.from_numpy(wz.s.view(np.int16)).to(dev).view(torch.float16), N, K, Gz)
            zkz = wq.wq_pack_int4_zeros(torch.from_numpy(synth.int4_zeros(N, K, Gz, seed + 2)).to(dev), N, K, Gz)
            outx = torch.empty((M, N), dtype=torch.float16, device=dev)
            byts = N * K // 2 + (K // Gz) * N * 3 + M * K * 2 + M * N * 2
            for op in ("w4a16_zp", "w4a16"):
                opid = wq.WQ_OP_W4A16_ZP if op == "w4a16_zp" else wq.WQ_OP_W4A16
                plan = wq.get_plan(opid, wq.WQ_F16, M, N, K, Gz)
                wsx = torch.zeros(plan["ws_bytes"] + 16, dtype=torch.uint8, device=dev)
                if op == "w4a16_zp":
                    call = lambda w=wkz: wq.wq_gemm_w4a16_zp(Ax, w, skz, zkz, N, K, Gz, out=outx, ws=wsx)
                else:
                    call = lambda w=wkz: wq.wq_gemm_w4a16(Ax, w, skz, N, K, Gz, out=outx, ws=wsx)
                us = time_call(call)
                ob = byts if op == "w4a16_zp" else byts - (K // Gz) * N
                extra = {"G": Gz, "kernel": plan["kernel"]}
                if M <= 16:
                    copies = [wkz] + [wkz.clone() for _ in range(n_copies(N * K // 2) - 1)]
                    extra.update(graph_fields(graph_us([(lambda w=w: call(w)) for w in copies]), ob))
                    del copies
                entry(op, M, N, K, "f16", us, ob, extra, into=zero_point)
                del wsx
            del Ax, wkz, skz, zkz, outx
        # codebook INT4 (NF4-style table) and INT2 W2A16: the register decode kernels at
        # M <= 16 (codebook: fp16 activations; INT2: G >= 64), the tile kernels above
        for (M, N, K, Gc) in [(16, 4096, 4096, 128), (4096, 4096, 4096, 128), (8192, 8192, 8192, 128)]:
            seed = 7000 + M
            Ax = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.int16)).to(dev).view(torch.float16)
            outx = torch.empty((M, N), dtype=torch.float16, device=dev)
            io = M * K * 2 + M * N * 2 + (K // Gc) * N * 2
            wc = synth.int4_weights(N, K, Gc, seed + 1)
            s_dev = torch.from_numpy(wc.s.view(np.int16)).to(dev).view(torch.float16)
            wkc, skc = wq.wq_pack_int4(torch.from_numpy(wc.w).to(dev), s_dev, N, K, Gc)
            lut = torch.from_numpy(synth.normal_quantile_codebook().view(np.int16)).to(dev).view(torch.float16)
            plan = wq.get_plan(wq.WQ_OP_W4A16_LUT, wq.WQ_F16, M, N, K, Gc)
            wsx = torch.zeros(plan["ws_bytes"] + 16, dtype=torch.uint8, device=dev)
            call = lambda w=wkc: wq.wq_gemm_w4a16_lut(Ax, w, skc, lut, N, K, Gc, out=outx, ws=wsx)
            us = time_call(call)
            extra = {"G": Gc, "kernel": plan["kernel"]}
            if M <= 16:
                copies = [wkc] + [wkc.clone() for _ in range(n_copies(N * K // 2) - 1)]
                extra.update(graph_fields(graph_us([(lambda w=w: call(w)) for w in copies]), N * K // 2 + io + 32))
                del copies
            entry("w4a16_lut", M, N, K, "f16", us, N * K // 2 + io + 32, extra, into=codebook_int2)
            del wkc, skc, wsx
            w2 = synth.int2_weights(N, K, Gc, seed + 2)
            w2d = torch.from_numpy(w2.w).to(dev)
            sk2 = wq.wq_pack_int2_scales(torch.from_numpy(w2.s.view(np.int16)).to(dev).view(torch.float16), N, K, Gc)
            plan = wq.get_plan(wq.WQ_OP_W2A16, wq.WQ_F16, M, N, K, Gc)
            wsx = torch.zeros(plan["ws_bytes"] + 16, dtype=torch.uint8, device=dev)
            call = lambda w=w2d: wq.wq_gemm_w2a16(Ax, w, sk2, N, K, Gc, out=outx, ws=wsx)
            us = time_call(call)
            extra = {"G": Gc, "kernel": plan["kernel"]}
            if M <= 16:
                copies = [w2d] + [w2d.clone() for _ in range(n_copies(N * K // 4) - 1)]
                extra.update(graph_fields(graph_us([(lambda w=w: call(w)) for w in copies]), N * K // 4 + io))
                del copies
            entry("w2a16", M, N, K, "f16", us, N * K // 4 + io, extra, into=codebook_int2)
            del Ax, w2d, sk2, wsx, outx, s_dev
        del flush

    # ---------------- quantiser extra: fp16 W (11008 x 4096) -> INT4 codes + fp16 scales
    quantiser = []
    if not args.skip_prefill:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        for Gq in (32, 128):
            Nq, Kq = 11008, 4096
            Wq = torch.randn((Nq, Kq), generator=torch.Generator().manual_seed(77), dtype=torch.float32)
            Wq = (Wq * 0.02).to(torch.float16).to(dev)
            times = []
            with torch.cuda.stream(stream):
                for it in range(3 + 10):
                    flush.fill_(it & 0xFF)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    wq.wq_quantize_int4(Wq, Gq)
                    b.record(stream)
                    times.append((a, b))
            torch.cuda.synchronize(dev)
            us = statistics.median([a.elapsed_time(b) * 1e3 for a, b in times[3:]])
            qbytes = Nq * Kq * 2 + Nq * Kq // 2 + (Kq // Gq) * Nq * 2
            quantiser.append({"N": Nq, "K": Kq, "G": Gq, "us": round(us, 2), "GB/s": round(qbytes / (us * 1e-6) / 1e9, 1),
                              "frac_hbm": round(qbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)})
        del flush

    # ---------------- end to end through the public API (pinned host buffers)
    e2e_steps = max(3, min(args.steps, 50))
    host_in = [[torch.empty(A.shape, dtype=A.dtype, pin_memory=True).copy_(A.cpu()) for (_, _, _, A, *_r) in s]
               for s in gemms]
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for (*_r, o) in s] for s in gemms]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0])
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            r = i % ROTATING_SETS
            for j, (M, N, K, A, wk, sk, out) in enumerate(gemms[r]):
                A.copy_(host_in[r][j], non_blocking=True)
                wq.wq_gemm_w4a16(A, wk, sk, N, K, G, out=out, ws=ws)
                host_out[r][j].copy_(out, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_value = step_bytes * world / e2e_s / 1e9

    # ---------------- CPU baseline: the float64 oracle on the host cores (rank 0 only)
    cpu = None
    if rank == 0 and not args.skip_cpu:
        v, secs, cores, sample = cpu_oracle_decode(1.0 / 16, args.cpu_seconds)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}

    if rank != 0:
        return
    csum = clocks.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemms_per_step": launches_per_step, "algorithmic_bytes_per_step": step_bytes,
                   "l2": f"inputs larger than L2: {ROTATING_SETS} rotating weight sets "
                         f"({ROTATING_SETS * sum(wk.numel() + sk.numel() * 2 for (_, _, _, _, wk, sk, _) in gemms[0]) / 1e6:.0f} MB)",
                   "timed_region": "CUDA-graph replays of the 8-GEMM step", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "peak_source": f"{peaks_src} (MEASURED_PEAKS.json hbm_gbs)" if peaks_src == "measured"
                     else "fallback 6.8 TB/s",
                     "kernel": "wq_decode_mma_kernel<f16, NT=1|2, BK=256> (register-resident mma.sync, split-K)",
                     "achieved_from": "CUDA events on the launching stream over the timed region (graph "
                                      "replays; the decode kernel is the only kernel there): step bytes / step time",
                     "per_shape_graphs_GB/s": round(per_shape_rate, 1)},
        "per_gemm": sorted(per_gemm, key=lambda d: (d["M"], d["N"], d["K"])),
        "prefill": prefill,
        "quantiser": quantiser,
        "fp8_fp4": fp8_fp4,
        "zero_point": zero_point,
        "codebook_int2": codebook_int2,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4),
                "how": "per step: pinned-host->device copy of every A, wq_gemm_w4a16 via the Python binding, "
                       "device->pinned-host copy of every output, stream synchronize; host wall clock"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": csum,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """Runs one GEMM `--reps` times (a small, self-contained target for ncu)."""
    import torch
    import weight_only_quantized_tma_gb300 as wq
    from weight_only_quantized_tma_gb300 import build as wq_build
    from weight_only_quantized_tma_gb300 import synth
    wq_build.build()
    op, *dims = args.case.split(":")
    M, N, K = (int(x) for x in dims[:3])
    dev = torch.device("cuda", 0)
    seed = 7
    if op in ("w4a16", "lut"):
        Gc = int(dims[3]) if len(dims) > 3 else 128
        A = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.float16)).to(dev)
        w = synth.int4_weights(N, K, Gc, seed + 1)
        wk, sk = wq.wq_pack_int4(torch.from_numpy(w.w).to(dev), torch.from_numpy(w.s.view(np.float16)).to(dev),
                                 N, K, Gc)
        if op == "lut":
            lut = torch.from_numpy(synth.normal_quantile_codebook().view(np.int16)).to(dev).view(torch.float16)
            fn = lambda: wq.wq_gemm_w4a16_lut(A, wk, sk, lut, N, K, Gc)
        else:
            fn = lambda: wq.wq_gemm_w4a16(A, wk, sk, N, K, Gc)
    elif op == "int2":
        Gc = int(dims[3]) if len(dims) > 3 else 128
        A = torch.from_numpy(synth.activations(M, K, "f16", seed).view(np.float16)).to(dev)
        w = synth.int2_weights(N, K, Gc, seed + 1)
        w2d = torch.from_numpy(w.w).to(dev)
        sk2 = wq.wq_pack_int2_scales(torch.from_numpy(w.s.view(np.float16)).to(dev), N, K, Gc)
        fn = lambda: wq.wq_gemm_w2a16(A, w2d, sk2, N, K, Gc)
    elif op == "fp8":
        A = torch.from_numpy(synth.activations(M, K, "bf16", seed).view(np.int16)).view(torch.bfloat16).to(dev)
        w = synth.fp8_weights(N, K, seed + 1)
        wd = torch.from_numpy(w.w).to(dev)
        alpha = torch.tensor([w.scale], dtype=torch.float32, device=dev)
        fn = lambda: wq.wq_gemm_w8a16_fp8(A, wd, alpha)
    elif op == "fp4":
        A = torch.from_numpy(synth.activations(M, K, "bf16", seed).view(np.int16)).view(torch.bfloat16).to(dev)
        w = synth.fp4_weights(N, K, seed + 1)
        wd = torch.from_numpy(w.w).to(dev)
        sfk = wq.wq_pack_fp4_sf(torch.from_numpy(w.sf).to(dev), N, K)
        alpha = torch.tensor([w.alpha], dtype=torch.float32, device=dev)
        fn = lambda: wq.wq_gemm_bf16_fp4(A, wd, sfk, alpha)
    else:
        raise SystemExit(f"unknown case {args.case}")
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize(dev)
    print(json.dumps({"case": args.case, "reps": args.reps, "plan": wq.get_plan(
        {"w4a16": wq.WQ_OP_W4A16, "lut": wq.WQ_OP_W4A16_LUT, "int2": wq.WQ_OP_W2A16, "fp8": wq.WQ_OP_FP8,
         "fp4": wq.WQ_OP_FP4}[op],
        wq.WQ_F16 if op in ("w4a16", "lut", "int2") else wq.WQ_BF16, M, N, K, int(dims[3]) if len(dims) > 3 else 128)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", default=None,
                    help="profiling target: run one GEMM, e.g. w4a16:16:4096:4096:128, lut:M:N:K[:G], int2:M:N:K[:G], "
                         "fp8:M:N:K, fp4:M:N:K")
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
