"""Benchmark of the NF4-dequant-fused backward-A GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input: one
backward-A call on the workload's projection(s) (a grouped launch when the
workload has several).  The default workload is the full training step of a
Qwen2.5-1.5B-shaped model: 28 layers x 7 projections (q, k, v, o, gate, up,
down) at M=4096 tokens with fp32 grad_out, as one grouped call (196 problems,
10.7 TFLOP).  ``--layers L`` runs the first L layers only (for a profiler
capture of a small case).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise, timed with CUDA events on the launching stream.
The K steps replay a CUDA graph of G steps that rotates through enough input
sets (grad_out, NF4 weight, grad_A) to exceed the 129 MB L2, so no step reads
another step's inputs from L2.  Under torchrun every rank runs its own copy of
the workload (M-sharded data parallelism: independent token batches, no
collective on the data path); the reported time is the maximum over ranks.

The JSON line carries the device throughput (`value`), an end-to-end number
through the public API with host buffers (`e2e`), the roofline of the GEMM
kernel against MEASURED_PEAKS.json, the CPU oracle timed on a bounded sample
(`cpu_baseline`), and SM clocks sampled during the timed region.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (BF16, CONFIGS, DTYPE_NAMES, F32, FUSED, Problem, full_step,  # noqa
                       make_grad_out, make_weight)

L2_BYTES = 129 * 2**20
# Idle seconds before a kernel-alone timing that follows the timed steps: a
# step whose f16 pass runs beside the GEMM can hold the GPU at its power cap,
# and the lowered clock would otherwise carry over into the next timing.
KERNEL_PAUSE_S = 2.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workloads(layers: int | None = None) -> dict[str, list[Problem]]:
    w = {"q_proj": CONFIGS["q_proj"], "tiny": CONFIGS["tiny"],
         "up_proj": [CONFIGS["mlp"][0]], "down_proj": [CONFIGS["mlp"][1]],
         "mlp": CONFIGS["mlp"],
         "full_step": CONFIGS["full_step"] if layers is None else full_step(layers=layers)}
    for p in CONFIGS["large"]:
        w[p.name] = [p]
    return w


# Forward product C[M x N] = A[M x K] @ dequant(B_nf4[K x N]) (nf4_forward_ws):
# the same projections in the forward direction.  (M, N out, K in, A dtype,
# A std, B std, outliers, seed)
FWD_WORKLOADS = {
    "fwd_q_proj": (2048, 1536, 1536, F32, 1e-2, 0.02, False, 0),
    "fwd_up_proj": (4096, 8960, 1536, BF16, 1e-2, 0.02, True, 0),
    "fwd_down_proj": (4096, 1536, 8960, BF16, 1e-2, 0.02, True, 2),
    "fwd_large": (8191, 14336, 4096, F32, 1.0, 0.015, False, 0),
}


def describe(name: str, probs: list[Problem]) -> str:
    if len(probs) == 1:
        p = probs[0]
        return f"{name}: M={p.M} N={p.N} K={p.K} grad_out {DTYPE_NAMES[p.go_dtype]}"
    if name == "full_step":
        return (f"full_step: {len(probs) // 7} layers x 7 projections (q, k, v, o, gate, up, down; "
                f"hidden 1536, kv 256, intermediate 8960), M={probs[0].M} tokens, grad_out "
                f"{DTYPE_NAMES[probs[0].go_dtype]}, one grouped call")
    return f"{name}: {len(probs)} projections grouped, M={probs[0].M}"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it), then a barrier; the time
    itself with one rank.  `device` holds the reduction's tensor (a CUDA device
    under NCCL, the CPU under gloo)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (ctypes) every ~2 ms."""

    # clocks_event_reasons bits (nvml.h)
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._ok = False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._ok = True
        except OSError:
            pass

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and
                    self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0):
                self.samples.append((clk.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        if self._ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._ok:
            self._stop.set()
            self._t.join()

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = sorted({name for _, r in busy for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in busy), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(busy)}


# ---------------------------------------------------------------- our arm
def make_input_sets(probs, copies, dev, entry="plain"):
    import backward_gemm_gb300 as nb

    sets = []
    base_go = [make_grad_out(p) for p in probs]
    base_B = [make_weight(p) for p in probs]
    for c in range(copies):
        items = []
        for p, go, B in zip(probs, base_go, base_B):
            if p.go_dtype == F32:
                go_t = torch.from_numpy(go).to(dev)
            else:
                go_t = torch.from_numpy(go.view(np.int16)).to(dev).view(torch.bfloat16)
            w = nb.quantize(torch.from_numpy(B).to(dev))
            out = torch.empty((p.M, p.K), dtype=torch.float32, device=dev)
            items.append((go_t, w, out))
        if len(items) > 1:
            ws = (nb.batched_ws_workspace(items, dev) if entry == "ws"
                  else nb.batched_workspace(len(items), dev))
        elif entry == "ws":
            ws = nb.ws_workspace(probs[0].M, probs[0].N, dev)
        else:
            ws = None
        sets.append((items, ws))
    torch.cuda.synchronize()
    return sets, base_go


RUN_ENTRY = {"entry": "plain"}  # the entry point run_step uses (set by bench_ours)


def run_step(items, ws):
    """One step through the public API.  With the ws entry a single problem runs
    nf4_backward_a_ws and a group nf4_backward_a_batched_ws (f16 pre-passes, then
    the GEMM); otherwise nf4_backward_a_ex / nf4_backward_a_batched."""
    import backward_gemm_gb300 as nb

    if len(items) == 1:
        go, w, out = items[0]
        if ws is None:
            nb.backward_a(go, w, out=out)
        else:
            nb.backward_a_ws(go, w, ws, out=out)
    elif RUN_ENTRY["entry"] == "ws":
        nb.backward_a_batched_ws(items, ws)
    else:
        nb.backward_a_batched(items, ws)


def bench_ours(args, rank, world, dev):
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    if rank == 0:
        build()
    if world > 1:
        torch.distributed.barrier()
    build()
    nb.lib()

    probs = workloads(args.layers)[args.workload]
    flops = sum(p.flops for p in probs)
    alg_bytes = sum(p.algorithmic_bytes for p in probs)
    entry = args.entry if len(probs) > 1 or probs[0].M > SMALL_M_MAX else "plain"
    RUN_ENTRY["entry"] = entry
    per_set = sum(p.go_bytes + 4 * p.M * p.K + p.K * p.N // 2
                  + (2 * p.M * p.N if entry == "ws" else 0) for p in probs)
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    sets, host_go = make_input_sets(probs, copies, dev, entry)
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            run_step(*sets[i % copies])
        nb.check_error()
        # Graph of `copies` steps, one per input set.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(copies):
                run_step(*sets[i])
        graph.replay()
        stream.synchronize()

        K = args.steps
        full, rem = divmod(K, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                run_step(*sets[i])
            ev1.record(stream)
            ev1.synchronize()
        torch.cuda.synchronize(dev)
        ms = ev0.elapsed_time(ev1)
        nb.check_error()
    ms = max_over_ranks(ms, world, dev)

    ms_per_step = ms / K
    value = flops * K * world / (ms * 1e-3) / 1e12  # whole-job TFLOP/s

    # End to end through the public API with host buffers: pinned grad_out in,
    # grad_A out, copies inside the timed region.
    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(args, probs, host_go, sets, stream, dev, flops, world)

    # The dominant kernel alone: with the ws entry a step is the f16 pre-pass
    # plus the GEMM; the GEMM is timed by itself by handing it the f16 copy that
    # the steps left in each set's workspace (the f16 grad_out entry skips the
    # pre-pass), over the same rotating sets, with its own clock samples.  A
    # step's pass adds HBM traffic that can hold the GPU at its power cap; an
    # idle pause first keeps the lowered clock from carrying over.
    kernel_ms = None
    kernel_clocks = None
    if entry == "ws" and (len(probs) == 1 and probs[0].N % 8 == 0 or
                          len(probs) > 1 and all(p.M > SMALL_M_MAX for p in probs)):
        time.sleep(KERNEL_PAUSE_S)
        with ClockSampler(dev.index) as kclocks:
            if len(probs) == 1:
                kernel_ms = time_gemm_only(sets, probs[0], stream, dev, min(K, 200))
            else:
                kernel_ms = time_group_gemm_only(sets, probs, stream, dev, min(K, 200))
        kernel_clocks = kclocks.summary()

    peaks, peak_kind = load_peaks()
    long_run = ms > 1000.0
    peak_tf = peaks["bf16_tflops_sustained" if long_run else "bf16_tflops"]
    t_tensor = flops / (peak_tf * 1e12)
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    kern_ms = kernel_ms if kernel_ms is not None else ms_per_step
    if t_tensor >= t_hbm:
        achieved = flops / (kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf}
    else:
        achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    roof["traffic"] = traffic_for(args.workload)
    roof["peak_source"] = (f"{peak_kind} {'sustained' if long_run else 'burst'} bf16 "
                           "(f16 nominal rate = bf16)" if roof["bound"] == "tensor"
                           else f"{peak_kind} HBM copy")
    roof["kernel"] = kernel_names(probs, entry)
    roof["kernel_ms"] = kern_ms
    roof["timed"] = ("whole step" if kernel_ms is None else
                     "bwd_a_kernel alone (f16 grad_out entry, CUDA events, same rotating sets, "
                     f"after the timed steps and a {KERNEL_PAUSE_S:g} s pause)"
                     if len(probs) == 1 else
                     "grouped bwd_a_kernel launch alone (f16 grad_out read in place, CUDA events, "
                     f"same rotating sets, after the timed steps and a {KERNEL_PAUSE_S:g} s pause; "
                     "its descriptor-upload kernels, ~2 us each, included)")
    if kernel_clocks is not None:
        roof["clocks"] = kernel_clocks

    line = {
        "metric": "NF4 backward-A GEMM TFLOP/s and % of GB300 dense FP16 tensor/HBM roofline",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": describe(args.workload, probs), "problems": len(probs),
                   "gflop_per_step": flops / 1e9, "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": ("nf4_backward_a_ws" if len(probs) == 1 else "nf4_backward_a_batched_ws")
                            if entry == "ws" else (
                       "nf4_backward_a_ex" if len(probs) == 1 else "nf4_backward_a_batched"),
                   "parallelism": f"dp{world} (M-sharded replicas, no collective)"},
        "e2e": e2e,
        "roofline": roof,
        "gpu_launches": K * launches_per_step(probs, entry),
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(probs, budget_s=args.cpu_seconds)
    return line


def bench_forward(args, dev):
    """The forward product through nf4_forward_ws on rotating input sets beyond
    L2 (a CUDA graph of one step per set), its GEMM kernel alone (f16 A left in
    each set's workspace by the steps), the tensor roofline and the clocks."""
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    build()
    nb.lib()
    M, N, K, dt, a_std, b_std, outl, seed = FWD_WORKLOADS[args.workload]
    a_np = make_grad_out(Problem(M, K, N, dt, a_std, b_std, outl, seed))      # A [M, K]
    B_np = make_weight(Problem(M, N, K, dt, a_std, b_std, outl, seed + 1))    # B [K, N]
    a_bytes = M * K * (4 if dt == F32 else 2)
    per_set = a_bytes + 4 * M * N + K * N // 2 + 2 * M * K
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    sets = []
    for _ in range(copies):
        a_t = (torch.from_numpy(a_np).to(dev) if dt == F32
               else torch.from_numpy(a_np.view(np.int16)).to(dev).view(torch.bfloat16))
        w = nb.quantize(torch.from_numpy(B_np).to(dev))
        sets.append((a_t, w, torch.empty((M, N), device=dev), nb.fwd_workspace(M, K, dev)))
    stream = torch.cuda.Stream(device=dev)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            a_t, w, c, ws = sets[i % copies]
            nb.forward_ws(a_t, w, ws, out=c)
        nb.check_error()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for a_t, w, c, ws in sets:
                nb.forward_ws(a_t, w, ws, out=c)
        graph.replay()
        stream.synchronize()
        full, rem = divmod(steps, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                a_t, w, c, ws = sets[i]
                nb.forward_ws(a_t, w, ws, out=c)
            ev1.record(stream)
            ev1.synchronize()
        ms = ev0.elapsed_time(ev1)
        # The GEMM alone: its f16 A is in each set's workspace after the steps
        # (timed after an idle pause, KERNEL_PAUSE_S).
        runs = [(ws[: 2 * M * K].view(torch.float16).view(M, K), w, c, ws) for _, w, c, ws in sets]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        time.sleep(KERNEL_PAUSE_S)
        e0.record(stream)
        for i in range(steps):
            a16, w, c, ws = runs[i % copies]
            nb.forward_ws(a16, w, ws, out=c)
        e1.record(stream)
        e1.synchronize()
        kern_ms = e0.elapsed_time(e1) / steps
        nb.check_error()
    flops = 2 * M * N * K
    alg_bytes = a_bytes + K * N // 2 + 4 * N * (K // 64) + 4 * M * N
    peaks, peak_kind = load_peaks()
    peak_tf = peaks["bf16_tflops_sustained" if ms > 1000.0 else "bf16_tflops"]
    achieved = flops / (kern_ms * 1e-3) / 1e12
    return {
        "metric": "NF4 forward GEMM (C = A @ dequant(B)) TFLOP/s and % of GB300 dense FP16 tensor roofline",
        "value": flops * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"{args.workload}: M={M} N={N} K={K} A {DTYPE_NAMES[dt]}",
                   "gflop_per_step": flops / 1e9, "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": "nf4_forward_ws", "parallelism": "dp1 (M-sharded replicas, no collective)"},
        "e2e": None,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": None,
                     "peak_source": f"{peak_kind} bf16 (f16 nominal rate = bf16)",
                     "kernel": "bwd_a_kernel (forward orientation)", "kernel_ms": kern_ms,
                     "timed": "GEMM alone (f16 A entry, CUDA events, same rotating sets)"},
        "gpu_launches": steps * 2,
        "clocks": clocks.summary(),
    }


# The full step with the sibling projections fused (nf4_backward_a_fused_batched):
# per layer q/k/v summed into one grad_x (three parts), o, gate/up summed (two
# parts), down -- 112 problems for the 28 layers, the same 10.7 TFLOP as the
# 196-projection step, each part with the full step's seeded inputs.
FUSED_STEP_GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def fused_step_groups(layers: int):
    probs = full_step(layers=layers)
    by_name = {p.name: p for p in probs}
    out = []
    for layer in range(layers):
        for names in FUSED_STEP_GROUPS:
            out.append([by_name[f"L{layer}.{n}"] for n in names])
    return out


def bench_fused_step(args, dev):
    """nf4_backward_a_fused_batched over the fused full step on rotating input
    sets beyond L2 (a CUDA graph of one step per set), the grouped GEMM alone
    (the f16 operands the steps left in each set's workspace, read in place),
    the tensor roofline, the clocks."""
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    build()
    nb.lib()
    groups = fused_step_groups(args.layers or 28)
    flat = [p for g in groups for p in g]
    flops = sum(p.flops for p in flat)
    alg_bytes = sum(p.go_bytes + p.K * p.N // 2 + 4 * p.N * (p.K // 64) for p in flat) + \
        sum(4 * g[0].M * g[0].K for g in groups)
    base = {p.name: (make_grad_out(p), make_weight(p)) for p in flat}
    per_set = sum(p.go_bytes + p.K * p.N // 2 + 2 * p.M * p.N for p in flat) + \
        sum(4 * g[0].M * g[0].K for g in groups)
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    sets = []
    for _ in range(copies):
        items = []
        for g in groups:
            gos = [torch.from_numpy(base[p.name][0]).to(dev) for p in g]
            w = nb.stack_weights([nb.quantize(torch.from_numpy(base[p.name][1]).to(dev)) for p in g])
            items.append((gos, w, torch.empty((g[0].M, g[0].K), device=dev)))
        arr, keep, _ = nb._fused_array(items)
        n = int(nb.lib().nf4_backward_a_fused_batched_ws_bytes(arr, len(items)))
        sets.append((items, torch.empty(n, dtype=torch.uint8, device=dev)))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            nb.backward_a_fused_batched(*sets[i % copies])
        nb.check_error()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for items, ws in sets:
                nb.backward_a_fused_batched(items, ws)
        graph.replay()
        stream.synchronize()
        full, rem = divmod(steps, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                nb.backward_a_fused_batched(*sets[i])
            ev1.record(stream)
            ev1.synchronize()
        ms = ev0.elapsed_time(ev1)
        nb.check_error()
        # The grouped GEMM alone: each problem's f16 operand [M][sum N] is in
        # the workspace after the steps (descriptors first, then the copies in
        # problem order); given as one f16 part it is read in place.  Timed
        # after an idle pause (KERNEL_PAUSE_S), with its own clock samples.
        runs = []
        desc = (640 * len(groups) + 255) // 256 * 256
        for items, ws in sets:
            at = desc
            f16_items = []
            for gos, w, out in items:
                M, N = gos[0].shape[0], w.N
                n = 2 * M * N
                f16_items.append(([ws[at: at + n].view(torch.float16).view(M, N)], w, out))
                at += (n + 255) // 256 * 256
            runs.append((f16_items, ws))
        kern_steps = min(steps, 200)
        for i in range(3):
            nb.backward_a_fused_batched(*runs[i % copies])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        time.sleep(KERNEL_PAUSE_S)
        with ClockSampler(dev.index) as kclocks:
            e0.record(stream)
            for i in range(kern_steps):
                nb.backward_a_fused_batched(*runs[i % copies])
            e1.record(stream)
            e1.synchronize()
        kern_ms = e0.elapsed_time(e1) / kern_steps
        nb.check_error()
    peaks, peak_kind = load_peaks()
    peak_tf = peaks["bf16_tflops_sustained" if ms > 1000.0 else "bf16_tflops"]
    achieved = flops / (kern_ms * 1e-3) / 1e12
    return {
        "metric": "NF4 backward-A GEMM TFLOP/s and % of GB300 dense FP16 tensor/HBM roofline",
        "value": flops * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"full_step_fused: {len(groups) // 4} layers x (q+k+v, o, gate+up, "
                               f"down) = {len(groups)} grouped problems, M={groups[0][0].M}, "
                               "grad_out f32",
                   "gflop_per_step": flops / 1e9, "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": "nf4_backward_a_fused_batched", "parallelism": "dp1"},
        "e2e": None,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": traffic_for("full_step_fused"),
                     "peak_source": f"{peak_kind} bf16 (f16 nominal rate = bf16)",
                     "kernel": "to_f16_stream_kernel (beside) + bwd_a_kernel", "kernel_ms": kern_ms,
                     "timed": "grouped bwd_a_kernel launch alone (f16 operands read in place, "
                              f"after the timed steps and a {KERNEL_PAUSE_S:g} s pause)",
                     "clocks": kclocks.summary()},
        "gpu_launches": steps * (-(-len(groups) // DESCS_PER_UPLOAD) + 2),  # uploads, pass, GEMM
        "clocks": clocks.summary(),
    }


# Fused input gradient of sibling projections (nf4_backward_a_fused): q/k/v and
# gate/up of one layer at M = 4096, each part with its own seeded grad_out
# (fp32) and weight; the weights stacked along N.
def bench_fused(args, dev):
    """nf4_backward_a_fused on rotating input sets beyond L2 (a CUDA graph of one
    step per set), its GEMM alone (the pre-converted single call on the f16 A
    operand the steps left in each set's workspace), the tensor roofline, the
    clocks and the oracle's fused sum on a bounded sample."""
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    build()
    nb.lib()
    parts = FUSED[args.workload]
    M, K = parts[0].M, parts[0].K
    N = sum(p.N for p in parts)
    host_go = [make_grad_out(p) for p in parts]
    host_B = [make_weight(p) for p in parts]
    per_set = sum(p.go_bytes for p in parts) + 4 * M * K + K * N // 2 + 2 * M * N
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    sets = []
    for _ in range(copies):
        gos = [torch.from_numpy(g).to(dev) for g in host_go]
        w = nb.stack_weights([nb.quantize(torch.from_numpy(B).to(dev)) for B in host_B])
        sets.append((gos, w, torch.empty((M, K), device=dev), nb.ws_workspace(M, N, dev)))
    stream = torch.cuda.Stream(device=dev)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            gos, w, out, ws = sets[i % copies]
            nb.backward_a_fused(gos, w, ws, out=out)
        nb.check_error()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for gos, w, out, ws in sets:
                nb.backward_a_fused(gos, w, ws, out=out)
        graph.replay()
        stream.synchronize()
        full, rem = divmod(steps, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                gos, w, out, ws = sets[i]
                nb.backward_a_fused(gos, w, ws, out=out)
            ev1.record(stream)
            ev1.synchronize()
        ms = ev0.elapsed_time(ev1)
        # The GEMM alone: the f16 A operand [M, N] is in each set's workspace.
        runs = [(ws[: 2 * M * N].view(torch.float16).view(M, N), w, out, ws)
                for _, w, out, ws in sets]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        kern_steps = min(steps, 200)
        torch.cuda.synchronize(dev)
        time.sleep(KERNEL_PAUSE_S)  # after the steps: see KERNEL_PAUSE_S
        e0.record(stream)
        for i in range(kern_steps):
            a16, w, out, ws = runs[i % copies]
            nb.backward_a_ws(a16, w, ws, out=out)
        e1.record(stream)
        e1.synchronize()
        kern_ms = e0.elapsed_time(e1) / kern_steps
        nb.check_error()
    flops = 2 * M * N * K
    alg_bytes = sum(p.go_bytes for p in parts) + K * N // 2 + 4 * N * (K // 64) + 4 * M * K
    peaks, peak_kind = load_peaks()
    peak_tf = peaks["bf16_tflops_sustained" if ms > 1000.0 else "bf16_tflops"]
    achieved = flops / (kern_ms * 1e-3) / 1e12
    line = {
        "metric": "NF4 fused sibling-projection backward-A (grad_x = sum_p g_p @ dequant(B_p)^T) "
                  "TFLOP/s and % of GB300 dense FP16 tensor roofline",
        "value": flops * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"{args.workload}: M={M} K={K} parts N=" +
                               "+".join(str(p.N) for p in parts) + " grad_out f32",
                   "gflop_per_step": flops / 1e9, "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": "nf4_backward_a_fused", "parallelism": "dp1"},
        "e2e": None,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": traffic_for(args.workload),
                     "peak_source": f"{peak_kind} bf16 (f16 nominal rate = bf16)",
                     "kernel": "to_f16_group_kernel + bwd_a_kernel", "kernel_ms": kern_ms,
                     "timed": "bwd_a_kernel alone (f16 A operand entry, CUDA events, same rotating sets)"},
        "gpu_launches": steps * 2,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_fused(parts, host_go, host_B, args.cpu_seconds)
    return line


def cpu_baseline_fused(parts, host_go, host_B, budget_s: float = 15.0):
    """The oracle's fused sum as it stands on a bounded sample of rows (about
    50 GFLOP; dequantise, rounding and the product timed, quantise not)."""
    import oracle

    M, K = parts[0].M, parts[0].K
    N = sum(p.N for p in parts)
    qs = [oracle.quantize(B) for B in host_B]
    rows = max(1, min(M, int(5e10 / (2 * N * K))))
    t0 = time.perf_counter()
    bts = [oracle.dequantize_f16(s, d, K, p.N) for p, (d, s) in zip(parts, qs)]
    go16s = [oracle.round_operand(g[:rows], p.go_dtype) for p, g in zip(parts, host_go)]
    oracle.backward_a_fused_rows(go16s, bts, np.arange(rows, dtype=np.int32), want_bound=False)
    dt = time.perf_counter() - t0
    return {"value": 2 * rows * N * K / dt / 1e12, "unit": "TFLOP/s",
            "cores": oracle.max_threads(), "kind": "oracle", "seconds": dt,
            "sample": f"{rows} of {M} rows of the fused {M}x{N}x{K} product; fp64 sums; "
                      "dequantise + rounding + product timed, quantise not"}


# Dense weight gradient grad_B = A^T @ grad_C (nf4_gemm_backward_b), bf16 operands:
# a full q_proj-shaped weight gradient (compute bound) and a rank-16 adapter's
# gradient against the up projection's output width (HBM bound).  (M tokens,
# K rows of grad_B, N columns)
BWD_B_WORKLOADS = {"bwd_b_dense": (4096, 1536, 1536), "bwd_b_lora": (4096, 16, 8960)}


def bench_backward_b(args, dev):
    """nf4_gemm_backward_b on rotating input sets beyond L2 (a CUDA graph of one
    step per set), the roofline of the bound that applies (tensor or HBM), the
    clocks and the oracle on a bounded sample of output rows."""
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    build()
    nb.lib()
    M, K, N = BWD_B_WORKLOADS[args.workload]
    g = torch.Generator().manual_seed(0)
    a_h = (torch.randn(M, K, generator=g) * 0.5).to(torch.bfloat16)
    c_h = (torch.randn(M, N, generator=g) * 0.01).to(torch.bfloat16)
    per_set = 2 * M * (K + N) + 4 * K * N
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    wsb = int(nb.lib().nf4_gemm_backward_b_ws_bytes(M, K, N))
    sets = [(a_h.to(dev), c_h.to(dev), torch.empty((K, N), device=dev),
             torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)) for _ in range(copies)]
    stream = torch.cuda.Stream(device=dev)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            a, c, out, ws = sets[i % copies]
            nb.gemm_backward_b(a, c, ws, out=out)
        nb.check_error()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for a, c, out, ws in sets:
                nb.gemm_backward_b(a, c, ws, out=out)
        graph.replay()
        stream.synchronize()
        full, rem = divmod(steps, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                a, c, out, ws = sets[i]
                nb.gemm_backward_b(a, c, ws, out=out)
            ev1.record(stream)
            ev1.synchronize()
        ms = ev0.elapsed_time(ev1)
        nb.check_error()
    flops = 2 * M * K * N
    alg_bytes = 2 * M * (K + N) + 4 * K * N
    peaks, peak_kind = load_peaks()
    peak_tf = peaks["bf16_tflops_sustained" if ms > 1000.0 else "bf16_tflops"]
    step_s = ms * 1e-3 / steps
    splits = int(nb.lib().nf4_gemm_backward_b_splits(M, K, N, 76))
    if flops / (peak_tf * 1e12) >= alg_bytes / (peaks["hbm_gbs"] * 1e9):
        achieved = flops / step_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf,
                "peak_source": f"{peak_kind} bf16 {'sustained' if ms > 1000.0 else 'burst'}"}
    else:
        achieved = alg_bytes / step_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_kind} HBM copy"}
    roof.update({"traffic": traffic_for(args.workload),
                 "kernel": "backward_b_kernel" + (" + reduce_splits_kernel" if splits > 1 else ""),
                 "kernel_ms": ms / steps, "timed": "whole step"})
    line = {
        "metric": "Dense GemmBackwardB (grad_B = A^T @ grad_C) TFLOP/s and % of GB300 roofline",
        "value": flops * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"{args.workload}: M={M} tokens, K={K}, N={N}, bf16",
                   "gflop_per_step": flops / 1e9, "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "token_splits": splits,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": "nf4_gemm_backward_b", "parallelism": "dp1"},
        "e2e": None,
        "roofline": roof,
        "gpu_launches": steps * (2 if splits > 1 else 1),
        "clocks": clocks.summary(),
    }
    if not args.no_cpu:
        import oracle

        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
        rows = max(1, min(K, int(5e10 / (2 * M * N))))
        t0 = time.perf_counter()
        oracle.gemm_backward_b_rows(bits(a_h), bits(c_h), oracle.HALF_BF16,
                                    rows=np.arange(rows, dtype=np.int32), want_bound=False)
        dt_s = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 2 * M * N * rows / dt_s / 1e12, "unit": "TFLOP/s",
                                "cores": oracle.max_threads(), "kind": "oracle", "seconds": dt_s,
                                "sample": f"{rows} of {K} output rows; fp64 sums over {M} tokens"}
    return line


# Backward of RMS layer normalisation (rms_norm_backward), the step upstream of
# the projections' backward: rows = tokens, hidden = the model width.
RMSNORM_WORKLOADS = {"rmsnorm_bwd": (4096, 1536)}


def bench_rmsnorm(args, dev):
    """rms_norm_backward (dL/dx and dL/dgamma) on rotating input sets beyond L2;
    HBM roofline of its algorithmic bytes (x and g read, dL/dx written, r,
    gamma and dL/dgamma)."""
    import backward_gemm_gb300 as nb
    from backward_gemm_gb300.build import build

    build()
    nb.lib()
    rows, H = RMSNORM_WORKLOADS[args.workload]
    gen = torch.Generator().manual_seed(0)
    x = torch.randn(rows, H, generator=gen)
    gy = torch.randn(rows, H, generator=gen) * 1e-2
    gamma = 1.0 + 0.1 * torch.randn(H, generator=gen)
    rms = torch.sqrt((x.double() ** 2).mean(dim=1) + 1e-6).float()
    per_set = 12 * rows * H
    copies = max(2, min(16, -(-2 * L2_BYTES // per_set)))
    ws = torch.empty(max(int(nb.lib().rms_norm_backward_ws_bytes(rows, H)), 16),
                     dtype=torch.uint8, device=dev)
    sets = [(x.to(dev), gamma.to(dev), rms.to(dev), gy.to(dev), torch.empty(rows, H, device=dev),
             torch.empty(H, device=dev)) for _ in range(copies)]
    L = nb.lib()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    nbytes = ws.numel()

    def step(st):
        xs, gs, rs, ys, ox, og = st
        rc = L.rms_norm_backward(P(xs), P(gs), P(rs), P(ys), P(ox), P(og), rows, H, P(ws), nbytes,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if rc != 0:
            raise RuntimeError(f"rms_norm_backward failed: {rc}")

    stream = torch.cuda.Stream(device=dev)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(sets[i % copies])
        nb.check_error()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for st in sets:
                step(st)
        graph.replay()
        stream.synchronize()
        full, rem = divmod(steps, copies)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clocks:
            ev0.record(stream)
            for _ in range(full):
                graph.replay()
            for i in range(rem):
                step(sets[i])
            ev1.record(stream)
            ev1.synchronize()
        ms = ev0.elapsed_time(ev1)
        nb.check_error()
    alg_bytes = 12 * rows * H + 4 * rows + 8 * H
    gbs = alg_bytes * steps / (ms * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    return {
        "metric": "RMSNorm backward (dL/dx, dL/dgamma) GB/s and % of GB300 HBM roofline",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: rows={rows} hidden={H}",
                   "algorithmic_mb_per_step": alg_bytes / 1e6,
                   "l2": f"rotating {copies} input sets, {copies * per_set / 2**20:.0f} MiB > L2",
                   "timing": f"CUDA graph of {copies} steps, CUDA events",
                   "entry": "rms_norm_backward", "parallelism": "dp1"},
        "e2e": None,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_kind} HBM copy",
                     "kernel": "rows_kernel + gamma_kernel", "kernel_ms": ms / steps,
                     "timed": "whole step (two launches)"},
        "gpu_launches": steps * 2,
        "clocks": clocks.summary(),
    }


SMALL_M_MAX = 64      # the library's default few-token limit (nf4_set_small_m_max)
STREAM_MAX_JOBS = 256  # pass jobs the streamed f16 pass takes in one launch (kStreamMaxJobs)
DESCS_PER_UPLOAD = 48  # descriptors per upload kernel of a grouped launch
F16_JOBS_PER_LAUNCH = 64  # problems per grouped f16 pass (nf4_backward_a_batched_ws)


def time_gemm_only(sets, p, stream, dev, steps):
    """Average device time of the GEMM kernel alone (ms): nf4_backward_a_ws on
    the f16 copies the steps left in the sets' workspaces."""
    import backward_gemm_gb300 as nb

    runs = []
    for items, ws in sets:
        go, w, out = items[0]
        go16 = ws[: 2 * p.M * p.N].view(torch.float16).view(p.M, p.N)
        runs.append((go16, w, out, ws))
    with torch.cuda.stream(stream):
        for i in range(3):
            go16, w, out, ws = runs[i % len(runs)]
            nb.backward_a_ws(go16, w, ws, out=out)
        nb.check_error()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(steps):
            go16, w, out, ws = runs[i % len(runs)]
            nb.backward_a_ws(go16, w, ws, out=out)
        ev1.record(stream)
        ev1.synchronize()
        nb.check_error()
    return ev0.elapsed_time(ev1) / steps


def time_group_gemm_only(sets, probs, stream, dev, steps):
    """Average device time (ms) of a grouped step's GEMM launch alone:
    nf4_backward_a_batched_ws given, as f16 grad_out, the copies the steps left
    in each set's workspace (f16 input is read in place, so no pre-pass runs;
    only the descriptor uploads precede the GEMM)."""
    import backward_gemm_gb300 as nb

    count = len(probs)
    desc = (640 * count + 255) // 256 * 256  # descriptor area (nf4_backward_a_batched_ws_bytes)
    runs = []
    for items, ws in sets:
        at = desc
        f16_items = []
        for p, (go, w, out) in zip(probs, items):
            pitch = (p.N + 7) // 8 * 8
            n = 2 * p.M * pitch
            assert pitch == p.N, "f16 copies are read as [M, N] (N % 8 == 0)"
            f16_items.append((ws[at: at + n].view(torch.float16).view(p.M, p.N), w, out))
            at += (n + 255) // 256 * 256
        runs.append((f16_items, ws))
    with torch.cuda.stream(stream):
        for i in range(3):
            nb.backward_a_batched_ws(*runs[i % len(runs)])
        nb.check_error()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(steps):
            nb.backward_a_batched_ws(*runs[i % len(runs)])
        ev1.record(stream)
        ev1.synchronize()
        nb.check_error()
    return ev0.elapsed_time(ev1) / steps


def kernel_names(probs, entry="plain") -> str:
    """The library kernels one step launches: the few-token kernel for M <= 64,
    the pair kernel otherwise (after the f16 pre-pass with the ws entry)."""
    names = []
    if any(p.M <= SMALL_M_MAX for p in probs):
        names.append("small_m_kernel")
    if any(p.M > SMALL_M_MAX for p in probs):
        names.append("bwd_a_kernel")
        if entry == "ws":
            names.insert(0, "to_f16_kernel" if len(probs) == 1 else "to_f16_stream_kernel (beside)")
    return " + ".join(names)


def launches_per_step(probs, entry="plain") -> int:
    """Kernel launches of one step through the C ABI: a single problem is one
    launch (two with the ws entry: the f16 pre-pass and the GEMM); a grouped
    call launches one few-token kernel per problem with M <= 64, then the
    descriptor uploads and one grouped GEMM for the rest, plus with the ws
    entry the f16 pass: one launch beside the GEMM when the workspace has room
    for its bookkeeping (the bench's always has) and at most STREAM_MAX_JOBS
    problems need a copy, else F16_JOBS_PER_LAUNCH problems per launch before
    it."""
    if len(probs) == 1:
        return 2 if entry == "ws" and probs[0].M > SMALL_M_MAX else 1
    few = sum(1 for p in probs if p.M <= SMALL_M_MAX)
    rest = len(probs) - few
    if not rest:
        return few
    passes = 0
    if entry == "ws":
        passes = 1 if rest <= STREAM_MAX_JOBS else -(-rest // F16_JOBS_PER_LAUNCH)
    return few + -(-rest // DESCS_PER_UPLOAD) + passes + 1


def bench_e2e(args, probs, host_go, sets, stream, dev, flops, world):
    """The step end to end through the public API with host buffers: every step
    copies its grad_out in from pinned host memory, runs the backward-A call and
    copies grad_A back out.  Steps are pipelined the way an application would
    run them, over two device buffer sets and three streams: step i's copy-in,
    step i-1's compute and step i-2's copy-out overlap (the two copy directions
    use separate engines).  The time runs from the first copy-in to the last
    copy-out, divided by the number of steps."""
    import backward_gemm_gb300 as nb  # noqa: F401  (run_step uses it)

    bufs = [sets[0], sets[1 % len(sets)]]
    pinned_in = []
    for p, go in zip(probs, host_go):
        t = torch.from_numpy(go.view(np.int16) if p.go_dtype == BF16 else go)
        pinned_in.append(t.pin_memory())
    pinned_out = [torch.empty((p.M, p.K), dtype=torch.float32).pin_memory() for p in probs]
    h2d = sum(t.numel() * t.element_size() for t in pinned_in)
    d2h = sum(t.numel() * 4 for t in pinned_out)
    steps = max(4, min(args.steps, 50))
    # Copies of a step are spread over E streams per direction (problem j on
    # stream j % E), so that several copy engines serve each direction.
    E = 2 if len(probs) > 1 else 1
    s_in = [torch.cuda.Stream(device=dev) for _ in range(E)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(E)]
    ev_in = [[torch.cuda.Event() for _ in range(E)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(E)] for _ in range(2)]

    def issue(i):
        b = i % 2
        items, ws = bufs[b]
        for e in range(E):
            with torch.cuda.stream(s_in[e]):
                if i >= 2:
                    s_in[e].wait_event(ev_comp[b])   # step i-2 no longer reads these inputs
                for j in range(e, len(items), E):
                    go_d, hin = items[j][0], pinned_in[j]
                    dst = go_d.view(torch.int16) if go_d.dtype == torch.bfloat16 else go_d
                    dst.copy_(hin, non_blocking=True)
                ev_in[b][e].record(s_in[e])
        with torch.cuda.stream(stream):
            for e in range(E):
                stream.wait_event(ev_in[b][e])
                if i >= 2:
                    stream.wait_event(ev_out[b][e])  # step i-2's outputs are copied out
            run_step(items, ws)
            ev_comp[b].record(stream)
        for e in range(E):
            with torch.cuda.stream(s_out[e]):
                s_out[e].wait_event(ev_comp[b])
                for j in range(e, len(items), E):
                    pinned_out[j].copy_(items[j][2], non_blocking=True)
                ev_out[b][e].record(s_out[e])

    for i in range(2):
        issue(i)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s_in[0])
    for e in range(1, E):
        s_in[e].wait_event(ev0)
    for i in range(steps):
        issue(i)
    for e in range(1, E):
        s_out[0].wait_stream(s_out[e])
    ev1.record(s_out[0])
    ev1.synchronize()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps, world, dev)
    return {"value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": steps,
            "pipelined": f"copy-in ({E} streams), compute, copy-out ({E} streams), two buffer sets"}


def kernel_source_digest() -> str:
    """SHA-256 over the CUDA sources of the library (file names and code, with
    comments and blank lines removed: a change to a comment leaves the kernels,
    and so their counters, as they were).  The sources hold no string literal
    with a comment marker."""
    import hashlib
    import re

    csrc = os.path.join(ROOT, "backward_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
            h.update(name.encode())
            h.update(code.encode())
    return h.hexdigest()


def traffic_for(workload: str):
    """DRAM bytes (read + write) per launch of this workload's kernel, from the
    committed ncu summary, or null when there is none or when the kernel sources
    changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_sha256") != kernel_source_digest():
        return None
    entry = t.get("workloads", {}).get(workload)
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- oracle (CPU) arm
def cpu_baseline(probs, budget_s: float = 15.0, rows_per_problem: int | None = None):
    """The CPU oracle as it stands, on a bounded sample: for each of the first
    seven problems a slice of its rows, up to about 120 GFLOP of fp64 work
    each (dequantise, operand rounding and the product timed)."""
    import oracle

    threads = oracle.max_threads()
    t_total = 0.0
    done_flops = 0
    rows_total = 0
    sample_desc = []
    # The GPU step starts from quantised weights, so the oracle's quantisation
    # (a one-off per weight) is not timed; its dequantisation, the rounding of
    # grad_out and the fp64 product are.  The sample is the first seven
    # problems (for the full step: the first layer's projections, one of the
    # 28 identical layers).
    shapes = list(probs[:7])
    for p in shapes:
        go = make_grad_out(p)
        data, scales = oracle.quantize(make_weight(p))
        t0 = time.perf_counter()
        bt = oracle.dequantize_f16(scales, data, p.K, p.N)
        rows = rows_per_problem or max(1, min(p.M, int(1.2e11 / (2 * p.N * p.K)) or 1))
        go16 = oracle.round_operand(go[:rows], p.go_dtype)
        oracle.backward_a_rows(go16, bt, np.arange(rows, dtype=np.int32), want_bound=False)
        t_total += time.perf_counter() - t0
        done_flops += 2 * rows * p.N * p.K
        rows_total += rows
        sample_desc.append(f"{rows} of {p.M} rows of {p.M}x{p.N}x{p.K}")
        if t_total > budget_s:
            break
    more = ""
    if len(probs) > len(shapes):
        more = (f" ({rows_total} rows of the first {len(sample_desc)} of the {len(probs)} "
                f"problems, to a {budget_s:.0f} s budget)")
    return {"value": done_flops / t_total / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": t_total,
            "sample": "; ".join(sample_desc) + more
                      + "; fp64 sums; dequantise + rounding + product timed, quantise not"}


def bench_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    from oracle.build import build_oracle

    build_oracle()
    probs = workloads(args.layers)[args.workload]
    # The workload's distinct projection shapes (for the full step: the seven
    # projections of the first layer; the other layers repeat them), each
    # with its own seeded inputs; quantisation is a one-off per weight and is
    # not timed.
    shapes, seen = [], set()
    for p in probs:
        if (p.M, p.N, p.K, p.go_dtype) not in seen:
            seen.add((p.M, p.N, p.K, p.go_dtype))
            shapes.append(p)
    inputs = []
    for p in shapes:
        data, scales = oracle.quantize(make_weight(p))
        inputs.append((p, make_grad_out(p), data, scales))
    steps_done = 0
    # A bounded per-step sample: probe the oracle's rate on a few rows of each
    # shape, then size each step (the same number of rows of every shape) so
    # that warm-up plus timed steps take about a minute in total.
    probe = min(min(p.M for p in shapes), 8)
    t0 = time.perf_counter()
    for p, go, data, scales in inputs:
        bt = oracle.dequantize_f16(scales, data, p.K, p.N)
        oracle.backward_a_rows(oracle.round_operand(go[:probe], p.go_dtype), bt,
                               np.arange(probe, dtype=np.int32), want_bound=False)
    per_row = sum(2 * p.N * p.K for p in shapes)
    rate = probe * per_row / max(time.perf_counter() - t0, 1e-6)
    per_step_s = 60.0 / max(args.steps + args.warmup, 1)
    rows = max(1, min(min(p.M for p in shapes), int(rate * per_step_s / per_row)))

    def step():
        for p, go, data, scales in inputs:
            bt = oracle.dequantize_f16(scales, data, p.K, p.N)
            go16 = oracle.round_operand(go[:rows], p.go_dtype)
            oracle.backward_a_rows(go16, bt, np.arange(rows, dtype=np.int32), want_bound=False)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
        steps_done += 1
    dt = time.perf_counter() - t0
    flops = rows * per_row * steps_done
    value = flops / dt / 1e12
    sample = (f"{rows} rows of each of {len(shapes)} distinct projection shapes ("
              + ", ".join(f"{p.M}x{p.N}x{p.K}" for p in shapes)
              + ") per step (dequantise + rounding + fp64 rows)")
    return {"metric": "NF4 backward-A GEMM TFLOP/s and % of GB300 dense FP16 tensor/HBM roofline",
            "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(steps_done, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(args.workload, probs),
                       "parallelism": "host cores (OpenMP), rank 0 only"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def bench_reference_extra(args, rank, world):
    """The oracle arm of the forward and RMSNorm workloads: the CPU oracle as it
    stands on the host cores, each step a bounded sample of the workload's rows
    (about a minute for warm-up plus timed steps), on the ours arm's metric."""
    if rank != 0:
        return None
    import oracle
    from oracle.build import build_oracle

    build_oracle()
    per_step_s = 60.0 / max(args.steps + args.warmup, 1)
    if args.workload == "full_step_fused":
        groups = fused_step_groups(1)  # one layer: the other 27 repeat its shapes
        data = []
        for g in groups:
            qs = [oracle.quantize(make_weight(p)) for p in g]
            data.append((g, [make_grad_out(p) for p in g], qs))
        per_row = sum(2 * p.N * p.K for g in groups for p in g)

        def run_rows(rows):
            for g, gos, qs in data:
                bts = [oracle.dequantize_f16(sc, d, p.K, p.N) for p, (d, sc) in zip(g, qs)]
                oracle.backward_a_fused_rows([oracle.round_operand(x[:rows], p.go_dtype)
                                              for p, x in zip(g, gos)], bts,
                                             np.arange(rows, dtype=np.int32), want_bound=False)

        probe = 8
        t0 = time.perf_counter()
        run_rows(probe)
        rate = probe * per_row / max(time.perf_counter() - t0, 1e-6)
        rows = max(1, min(groups[0][0].M, int(rate * per_step_s / per_row)))

        def step():
            run_rows(rows)

        metric = "NF4 backward-A GEMM TFLOP/s and % of GB300 dense FP16 tensor/HBM roofline"
        unit = "TFLOP/s"
        workload = ("full_step_fused: 28 layers x (q+k+v, o, gate+up, down) = 112 grouped "
                    f"problems, M={groups[0][0].M}, grad_out f32")
        what = (f"of {groups[0][0].M} rows of each of the first layer's 4 fused problems per step "
                "(dequantise + rounding + fp64 fused rows)")
    elif args.workload in BWD_B_WORKLOADS:
        M, K, N = BWD_B_WORKLOADS[args.workload]
        g = torch.Generator().manual_seed(0)
        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
        a_b = bits((torch.randn(M, K, generator=g) * 0.5).to(torch.bfloat16))
        c_b = bits((torch.randn(M, N, generator=g) * 0.01).to(torch.bfloat16))
        probe = min(K, 2)
        t0 = time.perf_counter()
        oracle.gemm_backward_b_rows(a_b, c_b, oracle.HALF_BF16, rows=np.arange(probe, dtype=np.int32),
                                    want_bound=False)
        rate = 2 * probe * M * N / max(time.perf_counter() - t0, 1e-6)
        rows = max(1, min(K, int(rate * per_step_s / (2 * M * N))))

        def step():
            oracle.gemm_backward_b_rows(a_b, c_b, oracle.HALF_BF16,
                                        rows=np.arange(rows, dtype=np.int32), want_bound=False)

        metric = "Dense GemmBackwardB (grad_B = A^T @ grad_C) TFLOP/s and % of GB300 roofline"
        unit, per_row = "TFLOP/s", 2 * M * N
        workload = f"{args.workload}: M={M} tokens, K={K}, N={N}, bf16"
        what = f"of {K} output rows of the {M}-token weight gradient per step (fp64 sums)"
    elif args.workload in FUSED:
        parts = FUSED[args.workload]
        M, K = parts[0].M, parts[0].K
        N = sum(p.N for p in parts)
        gos = [make_grad_out(p) for p in parts]
        qs = [oracle.quantize(make_weight(p)) for p in parts]
        probe = 8
        t0 = time.perf_counter()
        bts = [oracle.dequantize_f16(s, d, K, p.N) for p, (d, s) in zip(parts, qs)]
        oracle.backward_a_fused_rows([oracle.round_operand(g[:probe], p.go_dtype)
                                      for p, g in zip(parts, gos)], bts,
                                     np.arange(probe, dtype=np.int32), want_bound=False)
        rate = 2 * probe * N * K / max(time.perf_counter() - t0, 1e-6)
        rows = max(1, min(M, int(rate * per_step_s / (2 * N * K))))

        def step():
            b = [oracle.dequantize_f16(s, d, K, p.N) for p, (d, s) in zip(parts, qs)]
            oracle.backward_a_fused_rows([oracle.round_operand(g[:rows], p.go_dtype)
                                          for p, g in zip(parts, gos)], b,
                                         np.arange(rows, dtype=np.int32), want_bound=False)

        metric = ("NF4 fused sibling-projection backward-A (grad_x = sum_p g_p @ dequant(B_p)^T) "
                  "TFLOP/s and % of GB300 dense FP16 tensor roofline")
        unit, per_row = "TFLOP/s", 2 * N * K
        workload = (f"{args.workload}: M={M} K={K} parts N=" + "+".join(str(p.N) for p in parts)
                    + " grad_out f32")
        what = f"of {M} rows of the fused {M}x{N}x{K} product per step (dequantise + rounding + fp64 rows)"
    elif args.workload in FWD_WORKLOADS:
        M, N, K, dt, a_std, b_std, outl, seed = FWD_WORKLOADS[args.workload]
        a = make_grad_out(Problem(M, K, N, dt, a_std, b_std, outl, seed))
        data, scales = oracle.quantize(make_weight(Problem(M, N, K, dt, a_std, b_std, outl, seed + 1)))
        probe = min(M, 8)
        t0 = time.perf_counter()
        bt = oracle.dequantize_f16(scales, data, K, N)
        oracle.forward_rows(oracle.round_operand(a[:probe], dt), bt,
                            np.arange(probe, dtype=np.int32), want_bound=False)
        rate = 2 * probe * N * K / max(time.perf_counter() - t0, 1e-6)
        rows = max(1, min(M, int(rate * per_step_s / (2 * N * K))))

        def step():
            b = oracle.dequantize_f16(scales, data, K, N)
            oracle.forward_rows(oracle.round_operand(a[:rows], dt), b,
                                np.arange(rows, dtype=np.int32), want_bound=False)

        metric = "NF4 forward GEMM (C = A @ dequant(B)) TFLOP/s and % of GB300 dense FP16 tensor roofline"
        unit, per_row = "TFLOP/s", 2 * N * K
        workload = f"{args.workload}: M={M} N={N} K={K} A {DTYPE_NAMES[dt]}"
        what = f"of {M} rows of {M}x{N}x{K} per step (dequantise + rounding + fp64 rows)"
    else:
        rows_all, H = RMSNORM_WORKLOADS[args.workload]
        gen = torch.Generator().manual_seed(0)
        x = torch.randn(rows_all, H, generator=gen).numpy()
        gy = (torch.randn(rows_all, H, generator=gen) * 1e-2).numpy()
        gamma = (1.0 + 0.1 * torch.randn(H, generator=gen)).numpy()
        rms = np.sqrt((x.astype(np.float64) ** 2).mean(axis=1) + 1e-6).astype(np.float32)
        probe = min(rows_all, 64)
        t0 = time.perf_counter()
        oracle.rms_norm.backward(x[:probe], gamma, rms[:probe], gy[:probe])
        rate = 12 * probe * H / max(time.perf_counter() - t0, 1e-6)
        rows = max(1, min(rows_all, int(rate * per_step_s / (12 * H))))

        def step():
            oracle.rms_norm.backward(x[:rows], gamma, rms[:rows], gy[:rows])

        metric = "RMSNorm backward (dL/dx, dL/dgamma) GB/s and % of GB300 HBM roofline"
        unit, per_row = "GB/s", 12 * H
        workload = f"{args.workload}: rows={rows_all} hidden={H}"
        what = f"of {rows_all} rows of {rows_all}x{H} per step (fp64 numpy)"
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt_s = time.perf_counter() - t0
    value = per_row * rows * args.steps / dt_s / (1e12 if unit == "TFLOP/s" else 1e9)
    return {"metric": metric, "impl": "reference", "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt_s * 1e3 / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": f"{rows} {what}"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="full_step",
                    choices=sorted(workloads()) + sorted(FWD_WORKLOADS) + sorted(RMSNORM_WORKLOADS)
                    + sorted(FUSED) + sorted(BWD_B_WORKLOADS) + ["full_step_fused"])
    ap.add_argument("--layers", type=int, default=None,
                    help="full_step only: run the first L of the 28 layers (a small case for a "
                         "profiler capture)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--entry", default="ws", choices=["plain", "ws"],
                    help="single-problem entry point: nf4_backward_a_ex, or nf4_backward_a_ws "
                         "(f16 pre-pass into a workspace, then the GEMM)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.workload in RMSNORM_WORKLOADS or args.workload in FWD_WORKLOADS or \
            args.workload in FUSED or args.workload in BWD_B_WORKLOADS or \
            args.workload == "full_step_fused":
        if args.impl == "reference":
            line = bench_reference_extra(args, rank, world)
        elif world > 1:
            line = {"impl": args.impl, "unavailable": "this workload is measured on one GPU"}
        else:
            dev = torch.device("cuda", local)
            torch.cuda.set_device(dev)
            line = (bench_rmsnorm if args.workload in RMSNORM_WORKLOADS else
                    bench_fused_step if args.workload == "full_step_fused" else
                    bench_fused if args.workload in FUSED else
                    bench_backward_b if args.workload in BWD_B_WORKLOADS else
                    bench_forward)(args, dev)
    elif args.impl == "reference":
        line = bench_reference(args, rank, world)
    else:
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        line = bench_ours(args, rank, world, dev)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
