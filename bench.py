#!/usr/bin/env python
"""Benchmark of the routed MoE expert layer on GB300: one step = routing
prologue + forward + backward of the whole layer through the C ABI.

Default workload: the DeepSeek-V3-shaped layer (T=8192 tokens, hidden 7168,
intermediate 2048, 256 experts, top-8; 22.5 GB of bf16 weights), synthetic
seeded inputs.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config v3]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Metric: useful FLOPs per second (padding excluded: 6*H*I per routed slot
forward, 12*H*I backward), also routed tokens/s and the fraction of the
measured BF16 dense peak.  Under torchrun each rank runs an independent
replica of the layer on its own GPU (the layer does not shard on one GPU;
scaling is weak) and the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_FLOP_FACTOR = {  # useful FLOPs per routed slot, in units of H*I
    "gemm_l1_fwd": 4.0, "gemm_l2_fwd": 2.0, "gemm_l2_dgrad": 2.0, "gemm_dw2": 2.0, "gemm_dw1": 4.0,
    "gemm_l1_dgrad": 4.0,
}


def gemm_alg_bytes(name: str, T: int, H: int, I: int, E: int, k: int) -> float:
    """Algorithmic DRAM bytes of one launch: the weights read once, a weight
    gradient written once, x / dY read once, the saved h written once (L1
    forward) and read once (L2 dgrad).  The row-ordered intermediates (a, o,
    dh, aw, dxp) and gathered rows are kernel traffic, not algorithmic bytes
    (gemm_planned_bytes)."""
    W1, W2 = 2.0 * E * H * 2 * I, 2.0 * E * I * H
    x = dY = 2.0 * T * H
    h = 2.0 * T * k * 2 * I
    return {
        "gemm_l1_fwd": W1 + x + h,
        "gemm_l2_fwd": W2,
        "gemm_l2_dgrad": W2 + dY + h,
        "gemm_dw2": dY + W2,
        "gemm_dw1": x + W1,
        "gemm_l1_dgrad": W1,
    }[name]


def gemm_planned_bytes(name: str, T: int, H: int, I: int, E: int, k: int) -> float:
    """DRAM bytes of one launch as the kernels are planned: every operand
    (intermediates included) read once and every output written once, routed
    rows unpadded (bf16 everywhere)."""
    tk = T * k
    W1, W2 = 2.0 * E * H * 2 * I, 2.0 * E * I * H
    x = dY = 2.0 * T * H
    h, a, rows_h = 2.0 * tk * 2 * I, 2.0 * tk * I, 2.0 * tk * H
    return {
        "gemm_l1_fwd": W1 + x + h + a,
        "gemm_l2_fwd": W2 + a + rows_h,
        "gemm_l2_dgrad": W2 + dY + h + a + h + a,
        "gemm_dw2": a + dY + W2,
        "gemm_dw1": x + h + W1,
        "gemm_l1_dgrad": W1 + h + rows_h,
    }[name]


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over the ranks (the job takes as long as its
    slowest replica); x itself with one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job rate: the units every rank processed in `steps` steps over
    the job's time (the maximum over ranks), per second."""
    return world * units_per_rank_step * steps / (ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return PEAKS_FALLBACK, "fallback"


# the sources that define the grouped-GEMM kernels whose DRAM traffic
# profiles/traffic.json records; a change to any of them voids the record
GEMM_SOURCES = ("gemm_common.cuh", "grouped_gemm_2sm.cuh", "wgrad_pair.cuh", "ptx.cuh", "moe_internal.h",
                "gemm_fwd.cu", "gemm_dgrad.cu", "gemm_wgrad.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "routed_grouped_gemm_routing_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle
def oracle_sample(shape, inputs, n_tok, n_exp=1, seed=0, clamp=0.0):
    """Host copies of a bounded sample of the workload for the CPU oracle:
    n_tok tokens (forward, dx, d topk_weights) and the weight gradients of
    n_exp experts taken at evenly spaced quantiles of the expert load (the
    median one when n_exp = 1).  n_tok >= T: the whole problem (every token
    and every expert).  Returns (callable running it, useful FLOPs,
    description)."""
    import numpy as np
    import torch

    import oracle
    from routed_grouped_gemm_routing_gb300.workloads import bf16_bits

    E, k, H, I = shape.E, shape.k, shape.H, shape.I
    dev = inputs["x"].device
    idx_all = inputs["topk_idx"].cpu().numpy()
    valid = (idx_all >= 0) & (idx_all < E)
    counts = np.bincount(idx_all[valid].ravel(), minlength=E)
    whole = n_tok >= shape.T
    if whole:
        toks = np.arange(shape.T)
        exps = np.arange(E)
    else:
        rng = np.random.default_rng(seed)
        toks = np.sort(rng.choice(shape.T, size=n_tok, replace=False))
        order = np.argsort(counts, kind="stable")
        exps = np.unique(order[[int((q + 0.5) * E / n_exp) for q in range(n_exp)]])

    def sub(ids):
        remap = np.full(E, -1, np.int64)
        remap[ids] = np.arange(len(ids))
        return remap

    idx = idx_all[toks].astype(np.int64)
    vt = (idx >= 0) & (idx < E)
    involved = np.unique(idx[vt])
    idx_t = np.where(vt, sub(involved)[np.clip(idx, 0, E - 1)], -1).astype(np.int32)
    it, tt = torch.as_tensor(involved, device=dev), torch.as_tensor(toks, device=dev)
    W1t, W2t = bf16_bits(inputs["W1"][it]), bf16_bits(inputs["W2"][it])
    xt, dYt = bf16_bits(inputs["x"][tt]), bf16_bits(inputs["dY"][tt])
    wt = inputs["topk_w"][tt].cpu().numpy().astype(np.float32)
    idx_e = np.where(valid, sub(exps)[np.clip(idx_all, 0, E - 1)], -1).astype(np.int32)
    et = torch.as_tensor(exps, device=dev)
    W1e, W2e = bf16_bits(inputs["W1"][et]), bf16_bits(inputs["W2"][et])
    xa, dYa = bf16_bits(inputs["x"]), bf16_bits(inputs["dY"])
    wa = inputs["topk_w"].cpu().numpy().astype(np.float32)

    def run():
        oracle.forward(xt, W1t, W2t, idx_t, wt, clamp=clamp)
        oracle.backward_tokens(xt, W1t, W2t, idx_t, wt, dYt, clamp=clamp)
        oracle.backward_experts(xa, W1e, W2e, idx_e, wa, dYa, clamp=clamp)

    slots = int(vt.sum())
    rows = int(counts[exps].sum())
    flops = 6.0 * H * I * slots + 6.0 * H * I * slots + 6.0 * H * I * rows
    if whole:
        desc = (f"the whole layer ({shape.T} tokens, {slots} routed slots, {E} experts) forward and backward; "
                f"oracle FP32")
    else:
        desc = (f"{len(toks)} tokens ({slots} routed slots): forward, dx, d topk_weights; plus dW1/dW2 of "
                f"{len(exps)} experts at load quantiles ({rows} rows); oracle FP32, useful FLOPs counted as in "
                f"the metric")
    return run, flops, desc


def time_oracle(shape, inputs, n_tok, n_exp, seconds, seed=0, clamp=0.0):
    """The oracle on a bounded sample, repeated until `seconds` have passed
    (at least once); its rate scaled to the whole step."""
    import oracle

    oracle.build()
    run, flops, desc = oracle_sample(shape, inputs, n_tok=n_tok, n_exp=n_exp, seed=seed, clamp=clamp)
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    rate = flops * reps / dt
    step_flops = shape.flops_forward() + shape.flops_backward()
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "host_cores_available": cpu_cores(), "kind": "oracle", "sample": f"{reps} x ({desc})",
            "seconds": dt, "extrapolated_full_step_s": step_flops / rate,
            "extrapolated_note": "the whole layer step at the sample's FLOP rate (extrapolated, not run)"}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


METRIC = "MoE layer fwd+bwd TFLOP/s (useful FLOPs) & routed tokens/s; % of GB300 BF16 dense peak"


def config_dict(shape, world, activation_clamp=0.0):
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    label = " (DeepSeek-V3-shaped expert layer)" if shape.name == "v3" else ""
    out = {"workload": f"{shape.name}: T={T} H={H} I={I} E={E} k={k}{label}",
           "T": T, "H": H, "I": I, "E": E, "k": k, "block_m": 128,
           "l2": "inputs larger than L2 (weights alone are many times the 129 MB L2)",
           "parallelism": "replicas" if world > 1 else "single GPU"}
    if activation_clamp > 0:
        out["activation_clamp"] = activation_clamp
    return out


# -------------------------------------------------------------- main arms
def run_reference(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from routed_grouped_gemm_routing_gb300.workloads import CONFIGS, make_layer_inputs

    shape = CONFIGS[args.config]
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inputs = make_layer_inputs(shape, seed=args.seed, device=dev)
    run, flops, desc = oracle_sample(shape, inputs, n_tok=args.ref_tokens, seed=args.seed,
                                     clamp=args.activation_clamp)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": config_dict(shape, args.gpus, args.activation_clamp),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


FWD_KERNELS = ("route_hist", "route_scan", "route_place", "gemm_l1_fwd", "gemm_l2_fwd", "combine_fwd")
# the other workloads (tiny, V2-Lite-, wide- and skewed-V3-shaped layers),
# timed after the headline one, one at a time
# (each one's buffers are freed before the next is drawn): (name, config,
# backward, timed steps, oracle sample tokens, oracle sample experts)
OTHER_CONFIGS = (("tiny", "tiny", True, 100, 64, 0), ("v2lite", "v2lite", True, 20, 32, 2),
                 ("wide_fwd", "wide", False, 10, 8, 1), ("wide", "wide", True, 10, 8, 1),
                 ("skew", "skew", True, 10, 16, 1))


def roofline_of(name, shape, avg_ms, peaks, peaks_src, config_key):
    """The kernel's roofline object: algorithmic bytes (or FLOPs) per launch
    over its average live duration, against the HBM roof below the ridge
    point of the measured peaks and the sustained tensor roof above it."""
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    flops = GEMM_FLOP_FACTOR[name] * H * I * shape.slots
    nbytes = gemm_alg_bytes(name, T, H, I, E, k)
    sec = avg_ms / 1e3
    ridge = float(peaks["bf16_tflops_sustained"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            ent = json.load(f).get(config_key, {}).get(name)
        if ent and ent.get("source_hash") == kernel_source_hash():
            traffic = ent["bytes_per_launch"]
    if flops / nbytes < ridge:
        achieved, peak = nbytes / sec / 1e9, float(peaks["hbm_gbs"])
        r = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak, "unit": "GB/s",
             "frac": achieved / peak, "traffic": traffic, "peak_source": f"hbm_gbs ({peaks_src}, copy bandwidth)"}
    else:
        achieved, peak = flops / sec / 1e12, float(peaks["bf16_tflops_sustained"])
        r = {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
             "frac": achieved / peak, "traffic": traffic,
             "peak_source": f"bf16_tflops_sustained ({peaks_src}); burst {float(peaks['bf16_tflops']):.1f}"}
    r.update({"algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
              "planned_bytes_per_launch": gemm_planned_bytes(name, T, H, I, E, k),
              "arithmetic_intensity": flops / nbytes, "ridge_flop_per_byte": ridge,
              "achieved_tflops": flops / sec / 1e12, "achieved_gbs": nbytes / sec / 1e9})
    return r


class LayerBench:
    """Device buffers of one workload and its timed steps (prologue +
    forward, and backward unless forward-only) through the C ABI."""

    def __init__(self, shape, dev, seed, activation_clamp=0.0, backward=True):
        from routed_grouped_gemm_routing_gb300.layer import MoEWorkspace
        from routed_grouped_gemm_routing_gb300.workloads import make_layer_inputs

        import torch

        self.shape, self.backward = shape, backward
        T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
        self.inp = make_layer_inputs(shape, seed=seed, device=dev, with_grad_out=backward)
        self.ws = MoEWorkspace(T, H, I, E, k, device=dev, activation_clamp=activation_clamp)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        if backward:
            self.dx = torch.empty_like(self.y)
            self.dW1 = torch.empty_like(self.inp["W1"])
            self.dW2 = torch.empty_like(self.inp["W2"])
            self.dw = torch.empty(T, k, dtype=torch.float32, device=dev)

    def step(self):
        from routed_grouped_gemm_routing_gb300 import binding as B

        s, inp, ws = self.ws.shape, self.inp, self.ws
        B.moe_route_prologue(s, inp["topk_idx"], ws.route)
        B.moe_forward(s, inp["x"], inp["W1"], inp["W2"], inp["topk_w"], ws.route, ws.saved, self.y)
        if self.backward:
            B.moe_backward(s, inp["dY"], inp["x"], inp["W1"], inp["W2"], inp["topk_w"], ws.route, ws.saved,
                           ws.bwd, self.dx, self.dW1, self.dW2, self.dw)

    def check_status(self, when):
        from routed_grouped_gemm_routing_gb300 import binding as B

        status = B.moe_read_status(self.ws.shape, self.ws.route)
        if status[B.STATUS_FLAGS] != 0:
            raise RuntimeError(f"kernel status flags {status[B.STATUS_FLAGS]:#x} {when}")

    def timed(self, steps, warmup, world, dev, clock_index):
        """Warm-up, then `steps` steps between CUDA events on the launching
        stream (barrier + synchronize on both sides), every launch bracketed
        by the library's trace events.  Returns (max-over-ranks ms, trace,
        clocks)."""
        import torch
        import torch.distributed as dist

        from routed_grouped_gemm_routing_gb300 import binding as B

        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        self.check_status("after warm-up")
        trace = B.KernelTrace(max_launches=16 * steps)
        clocks = ClockSampler(clock_index)
        clocks.start()
        time.sleep(0.3)
        stream = torch.cuda.current_stream()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        with trace:
            for _ in range(steps):
                self.step()
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clk = clocks.stop()
        self.check_status("in the timed region")
        return max_over_ranks(t0.elapsed_time(t1), world, dev), trace, clk

    def summary(self, ms, trace, steps, world, peaks, peaks_src, config_key):
        """Rates, per-kernel times, the forward / backward split and the
        dominant GEMM's roofline of a timed run."""
        shape = self.shape
        flops_step = shape.flops_forward() + (shape.flops_backward() if self.backward else 0.0)
        value = job_rate(flops_step, steps, world, ms) / 1e12
        per = {}
        for name, d in trace.durations_ms():
            per.setdefault(name, []).append(d)
        kernels = {n: {"launches": len(v), "avg_ms": statistics.mean(v), "total_ms": sum(v),
                       "share": sum(v) / ms} for n, v in per.items()}
        gemms = {n: v for n, v in kernels.items() if n in GEMM_FLOP_FACTOR}
        dom = max(gemms, key=lambda n: gemms[n]["total_ms"])
        return {
            "ms_per_step": ms / steps, "value": value, "unit": "TFLOP/s",
            "routed_tokens_per_s": job_rate(shape.slots, steps, world, ms),
            "pct_bf16_peak_burst": 100.0 * value / world / float(peaks["bf16_tflops"]),
            "pct_bf16_peak_sustained": 100.0 * value / world / float(peaks["bf16_tflops_sustained"]),
            "forward_ms": sum(v["avg_ms"] for n, v in kernels.items() if n in FWD_KERNELS),
            "backward_ms": sum(v["avg_ms"] for n, v in kernels.items() if n not in FWD_KERNELS),
            "gpu_launches": int(trace.count), "launches_per_step": trace.count / steps,
            "kernels": kernels,
            "roofline": roofline_of(dom, shape, gemms[dom]["avg_ms"], peaks, peaks_src, config_key),
        }


def fp8_forward_times(shape, inp, ws, y, dev, peaks):
    """The FP8 forward (E4M3 input per token, E4M3 W1 and W2 per column, UE8M0
    scales per 32 elements of K, block-scaled MMA in both GEMMs, a quantized
    between them), timed beside the bf16 forward on the same inputs: an
    inference variant, not the layer step.  The weights are quantized once
    beforehand (a weight transform), timed on their own.  None when H or I is
    not a multiple of 128."""
    import torch

    from routed_grouped_gemm_routing_gb300 import binding as B

    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    if H % 128 or I % 128:
        return None
    xq = torch.empty(T, H, dtype=torch.uint8, device=dev)
    xsf = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
    w1q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
    w1sf = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device=dev)
    w2q = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
    w2sf = torch.empty(E * H * I // 32, dtype=torch.uint8, device=dev)

    def quantize_weights():
        B.moe_quantize_weights_fp8(ws.shape, inp["W1"], w1q, w1sf)
        B.moe_quantize_w2_fp8(ws.shape, inp["W2"], w2q, w2sf)

    quantize_weights()
    torch.cuda.synchronize()
    wtrace = B.KernelTrace(max_launches=2 * 3)
    with wtrace:
        for _ in range(3):
            quantize_weights()
    torch.cuda.synchronize()
    wq = {}
    for kn, d in wtrace.durations_ms():
        wq.setdefault(kn, []).append(d)
    wq_ms = {kn: statistics.median(v) for kn, v in wq.items()}

    def fwd_fp8():
        B.moe_quantize_fp8(ws.shape, inp["x"], xq, xsf)
        B.moe_forward_fp8(ws.shape, xq, xsf, w1q, w1sf, w2q, w2sf, inp["topk_w"], ws.route, ws.saved, y)

    def fwd_bf16():
        B.moe_forward(ws.shape, inp["x"], inp["W1"], inp["W2"], inp["topk_w"], ws.route, ws.saved, y)

    B.moe_route_prologue(ws.shape, inp["topk_idx"], ws.route)
    per = {}
    for name, fn in (("fp8", fwd_fp8), ("bf16", fwd_bf16)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ftrace = B.KernelTrace(max_launches=8 * 10)
        with ftrace:
            for _ in range(10):
                fn()
        torch.cuda.synchronize()
        kk = {}
        for kn, d in ftrace.durations_ms():
            kk.setdefault(kn, []).append(d)
        per[name] = {kn: statistics.median(v) for kn, v in kk.items()}
    tk = T * k
    q_bytes = T * H * 2 + T * H + T * H // 32
    l1_ms = per["fp8"]["gemm_l1_fwd_fp8"]
    l2_ms = per["fp8"]["gemm_l2_fwd_fp8"]
    # W1 and its scales, x and its scales, h (bf16), a (E4M3) and its scales
    l1_bytes = E * 2 * I * H * (1 + 1 / 32) + T * H * (1 + 1 / 32) + 2.0 * tk * 2 * I + tk * I * (1 + 1 / 32)
    # W2 and its scales, a and its scales, o (bf16)
    l2_bytes = E * H * I * (1 + 1 / 32) + tk * I * (1 + 1 / 32) + 2.0 * tk * H
    hbm = float(peaks["hbm_gbs"])
    out = {"forward_ms": sum(per["fp8"].values()), "bf16_forward_ms": sum(per["bf16"].values()),
           "kernels_ms": per["fp8"], "bf16_kernels_ms": per["bf16"],
           "quantize_gbs": q_bytes / (per["fp8"]["quantize_fp8"] / 1e3) / 1e9,
           "quantize_frac_of_hbm": q_bytes / (per["fp8"]["quantize_fp8"] / 1e3) / 1e9 / hbm,
           "l1_fp8_gbs": l1_bytes / (l1_ms / 1e3) / 1e9,
           "l1_fp8_frac_of_hbm": l1_bytes / (l1_ms / 1e3) / 1e9 / hbm,
           "l1_fp8_tflops": 4.0 * H * I * tk / (l1_ms / 1e3) / 1e12,
           "l2_fp8_gbs": l2_bytes / (l2_ms / 1e3) / 1e9,
           "l2_fp8_frac_of_hbm": l2_bytes / (l2_ms / 1e3) / 1e9 / hbm,
           "l2_fp8_tflops": 2.0 * H * I * tk / (l2_ms / 1e3) / 1e12,
           "forward_tflops": 6.0 * H * I * tk / (sum(per["fp8"].values()) / 1e3) / 1e12,
           "weight_quantize_ms": wq_ms,
           "note": "median of 10 runs of moe_quantize_fp8 + moe_forward_fp8 (and of moe_forward) on the "
                   "workload; both GEMMs multiply E4M3 operands (W1 and W2 quantized once beforehand, "
                   "weight_quantize_ms) with block-scaled tcgen05.mma, a quantized to E4M3 in the L1 "
                   "epilogue; not part of the step"}
    del w1q, w1sf, w2q, w2sf
    return out


def run_other_configs(args, dev, world, rank, peaks, peaks_src):
    """The other workloads (OTHER_CONFIGS) on this GPU, one after another; the
    V3-shaped headline's buffers are already freed."""
    import numpy as np
    import torch

    from routed_grouped_gemm_routing_gb300.workloads import CONFIGS

    out = {}
    for key, cname, backward, steps, n_tok, n_exp in OTHER_CONFIGS:
        shape = CONFIGS[cname]
        lb = LayerBench(shape, dev, args.seed + rank, backward=backward)
        ms, trace, clk = lb.timed(steps, max(3, args.warmup), world, dev, dev.index if world == 1 else
                                  int(os.environ.get("LOCAL_RANK", "0")))
        r = lb.summary(ms, trace, steps, world, peaks, peaks_src, cname)
        r["kernels_ms"] = {n: v["avg_ms"] for n, v in r.pop("kernels").items()}
        r.update({"config": config_dict(shape, world), "steps": steps, "clocks": clk,
                  "step": "prologue + forward + backward" if backward else "prologue + forward (forward only)"})
        counts = np.bincount(lb.inp["topk_idx"].flatten().cpu().numpy(), minlength=shape.E)
        r["expert_load"] = {"min": int(counts.min()), "mean": float(counts.mean()), "max": int(counts.max()),
                            "below_block_m": int(((counts > 0) & (counts < 128)).sum()),
                            "empty": int((counts == 0).sum()), "top5": sorted(counts.tolist())[-5:][::-1]}
        # the FP8 forward once per shape: on the forward-only line when there is one
        fwd_only = {c for _, c, b, _, _, _ in OTHER_CONFIGS if not b}
        if not args.no_fp8 and (not backward or cname not in fwd_only):
            r["fp8_forward"] = fp8_forward_times(shape, lb.inp, lb.ws, lb.y, dev, peaks)
        if rank == 0 and world == 1 and not args.no_cpu_baseline and backward:
            whole = n_exp == 0
            r["cpu_baseline"] = time_oracle(shape, lb.inp, n_tok=shape.T if whole else n_tok,
                                            n_exp=max(1, n_exp), seconds=2.0, seed=args.seed)
        out[key] = r
        del lb, trace
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from routed_grouped_gemm_routing_gb300 import binding as B
    from routed_grouped_gemm_routing_gb300 import build
    from routed_grouped_gemm_routing_gb300.layer import HostPipeline
    from routed_grouped_gemm_routing_gb300.workloads import CONFIGS

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    B.lib()
    peaks, peaks_src = load_peaks()

    shape = CONFIGS[args.config]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    lb = LayerBench(shape, dev, args.seed + rank, activation_clamp=args.activation_clamp)
    ms, trace, clk = lb.timed(args.steps, args.warmup, world, dev, dev.index if world == 1 else local)
    head = lb.summary(ms, trace, args.steps, world, peaks, peaks_src, args.config)
    inp, ws, y = lb.inp, lb.ws, lb.y
    flops_step = shape.flops_forward() + shape.flops_backward()

    # the same step captured once in a CUDA graph and replayed (every launch
    # of the step is capturable: no host synchronisation, no allocation)
    graph = None
    if not args.no_graph:
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            lb.step()
        torch.cuda.current_stream().wait_stream(gs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            lb.step()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record()
        for _ in range(args.steps):
            g.replay()
        gb.record()
        torch.cuda.synchronize()
        gms = ga.elapsed_time(gb) / args.steps
        graph = {"ms_per_step": gms, "value": flops_step / (gms / 1e3) / 1e12, "unit": "TFLOP/s",
                 "note": "the prologue + forward + backward step captured once and replayed"}
        del g

    # end to end through the public API, from pinned host buffers
    e2e = None
    if not args.no_e2e:
        host = {n: inp[n].cpu().pin_memory() for n in ("x", "topk_idx", "topk_w", "dY")}
        outs = {"y_h": torch.empty(T, H, dtype=torch.bfloat16).pin_memory(),
                "dx_h": torch.empty(T, H, dtype=torch.bfloat16).pin_memory(),
                "dw_h": torch.empty(T, k, dtype=torch.float32).pin_memory()}
        pipe = HostPipeline(ws, inp["W1"], inp["W2"], lb.dW1, lb.dW2)

        def e2e_step():
            pipe.submit(host["x"], host["topk_idx"], host["topk_w"], host["dY"], outs["y_h"], outs["dx_h"],
                        outs["dw_h"])

        for _ in range(max(1, args.warmup)):
            e2e_step()
        pipe.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(pipe.compute)
        pipe.up.wait_stream(pipe.compute)
        for _ in range(args.steps):
            e2e_step()
        pipe.synchronize()
        b.record(pipe.compute)
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b), world, dev)
        h2d = sum(host[n].numel() * host[n].element_size() for n in host)
        d2h = sum(outs[n].numel() * outs[n].element_size() for n in ("y_h", "dx_h", "dw_h"))
        e2e = {"value": job_rate(flops_step, args.steps, world, ems) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems / args.steps,
               "note": "x, topk_idx, topk_weights, dY copied in from pinned host memory and y, dx, "
                       "d topk_weights copied out every step (HostPipeline: uploads of step n+1 and downloads "
                       "of step n overlap the kernels); dW1/dW2 stay on the device"}
        del pipe

    # the router stage in front of the layer (logits -> top-k ids and weights
    # -> routing tables), timed on its own: it is not part of the layer step
    # the metric counts, which takes topk_idx / topk_weights as inputs
    router = None
    if not args.no_router:
        g = torch.Generator(device=dev)
        g.manual_seed(args.seed * 7919 + 11)
        logits = torch.randn(T, E, generator=g, device=dev, dtype=torch.float32)
        r_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        r_w = torch.empty(T, k, dtype=torch.float32, device=dev)
        r_route = torch.empty(max(ws.layout.route_bytes, 16), dtype=torch.uint8, device=dev)
        for _ in range(3):
            B.moe_router_topk(ws.shape, logits, r_idx, r_w, r_route)
        torch.cuda.synchronize()
        rtrace = B.KernelTrace(max_launches=2 * 20)
        with rtrace:
            for _ in range(20):
                B.moe_router_topk(ws.shape, logits, r_idx, r_w, r_route)
        torch.cuda.synchronize()
        rper = {}
        for name, d in rtrace.durations_ms():
            rper.setdefault(name, []).append(d)
        rk = {n: statistics.median(v) for n, v in rper.items()}
        r_bytes = T * E * 4 + T * k * 8  # logits read once, ids and weights written once
        router = {"ms": sum(rk.values()), "kernels_ms": rk,
                  "router_topk_gbs": r_bytes / (rk["router_topk"] / 1e3) / 1e9,
                  "router_topk_frac_of_hbm": r_bytes / (rk["router_topk"] / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                  "note": "median of 20 runs of moe_router_topk (router kernel + routing prologue) on the "
                          "workload's logits; not part of the layer step"}

    fp8 = None
    if not args.no_fp8:
        fp8 = fp8_forward_times(shape, inp, ws, y, dev, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(shape, inp, n_tok=args.cpu_tokens, n_exp=args.cpu_experts, seconds=args.cpu_seconds,
                          seed=args.seed, clamp=args.activation_clamp)

    del lb, inp, ws, y
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    others = None if args.no_configs else run_other_configs(args, dev, world, rank, peaks, peaks_src)

    if rank != 0:
        dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC,
        "value": head["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "forward_ms": head["forward_ms"], "backward_ms": head["backward_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded Gaussian inputs and weights, Gaussian-logit top-k routing)",
        "config": config_dict(shape, world, args.activation_clamp),
        "routed_tokens_per_s": head["routed_tokens_per_s"],
        "pct_bf16_peak_burst": head["pct_bf16_peak_burst"],
        "pct_bf16_peak_sustained": head["pct_bf16_peak_sustained"],
        "peaks_source": peaks_src,
        "clocks": clk,
        "gpu_launches": head["gpu_launches"],
        "launches_per_step": head["launches_per_step"],
        "kernels": head["kernels"],
        "roofline": head["roofline"],
        "e2e": e2e,
        "graph": graph,
        "cpu_baseline": cpu,
        "router": router,
        "fp8_forward": fp8,
        "configs": others,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="v3")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-router", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--activation-clamp", type=float, default=0.0,
                    help="SwiGLU input clamp c > 0 (0: none, the default workload)")
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--cpu-experts", type=int, default=2)
    ap.add_argument("--cpu-seconds", type=float, default=5.0)
    ap.add_argument("--ref-tokens", type=int, default=2)
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
