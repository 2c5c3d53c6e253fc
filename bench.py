#!/usr/bin/env python3
"""Benchmark of the fused decode kernels on GB300 (prints ONE JSON line on rank 0).

Default workload (one "step" = one pass of the whole hot path): the 32-layer decode MLP
step - per layer add-RMSNorm on [1, 4096] bf16 (eps 1e-5) then the SwiGLU-prologue
W4A16 down projection K=14336 N=4096 (group 128), seeded synthetic inputs (seed 3). Its
weights (972 MB) exceed the 129 MB L2, so no flush is needed between steps. The step
is captured once in a CUDA graph and replayed.

Reported:
  value      achieved GB/s = algorithmic bytes per step / device time per step
             (CUDA events around K replays on the launching stream, max over ranks)
  e2e        the same metric through the public API (DecodeStep.run_pinned) with the
             per-token inputs in pinned host memory: the transfer of x, residual and
             every layer's gate/up in, the 64 kernels, the transfer of x_L and the
             residual out (fd_copy kernels in the step's graph), all inside the timed
             region
  roofline   the dominant kernel (the GEMV) - its average launch duration from CUDA
             events around replays of a graph of the step's 32 GEMV launches alone
  cpu_baseline  the CPU oracle, single-threaded, on a bounded sample of the workload
  configs    every other workload configuration timed in the same process (one call per
             step, rotating input sets, CUDA graph): the small GEMV, the 8192 x 4096
             add-RMSNorm and the K=9216 N=2560 GEMV against the 70 % target, the batched
             M=64 product on the tensor-core and CUDA-core kernels, the residual-epilogue
             GEMV and the gate/up GEMV (--no-configs skips them)
  --impl reference  times the CPU oracle alone (the reference arm of this benchmark), on
             a bounded sample of the chosen workload; ms_per_step is one sample's time

Other workloads (--workload gemv_94mb | rmsnorm_big | gemv_small | batched_m64 |
gemv_residual | gate_up | nvfp4_qkv) time one call per step and rotate ceil(3 x L2 / bytes) input
sets so every step reads HBM; --workload fused_layer times 32 layers of add-RMSNorm +
gate/up GEMV + down GEMV with the residual epilogue as one graph; --workload
persistent_step [--layers L] times the decode step as one persistent cooperative launch
(fd_decode_mlp_step; the decode_step line reports it too, as persistent_step).
"""

from __future__ import annotations

import os

# The CPU oracle legs run single-threaded (set before numpy loads a BLAS).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np
import torch

REPO = Path(__file__).resolve().parent
METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) for SwiGLU-W4A16 GEMV + add-RMSNorm"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0
KERNEL_SOURCES = {
    # the M = 1 kernel the decode step runs (bulk-copy kernel, with the folded add-RMSNorm)
    # and the headers it uses
    "swiglu_w4a16_gemv_add_rmsnorm": ["csrc/fd_gemv_tma.cu", "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh",
                                      "csrc/fd_w4_unpack.cuh", "csrc/fd_internal.h"],
    "swiglu_w4a16_gemv": ["csrc/fd_gemv_tma.cu", "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh",
                          "csrc/fd_w4_unpack.cuh", "csrc/fd_internal.h"],
    "add_rmsnorm": ["csrc/fd_add_rmsnorm.cu", "csrc/fd_internal.h"],
    # the horizontal gate/up GEMV runs the same kernel's plain-activation form
    "w4a16_gate_up_gemv": ["csrc/fd_gemv_tma.cu", "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh",
                           "csrc/fd_w4_unpack.cuh", "csrc/fd_internal.h"],
    "nvfp4_scaled_mm": ["csrc/fd_nvfp4.cu", "csrc/fd_nvfp4_plan.h", "csrc/fd_tc.cuh", "csrc/fd_tma.cuh",
                        "csrc/fd_internal.h"],
    # the residual-add epilogue is the same bulk-copy kernel's residual form
    "swiglu_w4a16_gemv_residual": ["csrc/fd_gemv_tma.cu", "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh",
                                   "csrc/fd_w4_unpack.cuh", "csrc/fd_internal.h"],
    # the tensor-core GEMV of batched decode (M >= 16)
    "gemv_tc": ["csrc/fd_gemv_tc.cu", "csrc/fd_gemv_tc_plan.h", "csrc/fd_tc.cuh",
                "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh", "csrc/fd_w4_unpack.cuh",
                "csrc/fd_internal.h"],
    # the decode step as one persistent kernel
    "decode_step": ["csrc/fd_decode_step.cu", "csrc/fd_gemv_common.cuh", "csrc/fd_tma.cuh",
                    "csrc/fd_w4_unpack.cuh", "csrc/fd_internal.h"],
}


# ----------------------------------------------------------------------------- helpers

# The arithmetic each GEMV kernel computes in: the M = 1 and CUDA-core kernels encode the
# activation per 32-k slice as block-scaled int16 and take exact int32 dp2a dot products
# with the int4 weights; the tensor-core kernel multiplies bf16 operands into fp32.
DTYPE_DP2A = "int4 weights x block-scaled int16 activations: exact int32 dp2a dots, fp32 sums; bf16 in/out"
DTYPE_TC = "int4 weights dequantised to bf16 x bf16 activations on tcgen05, fp32 accumulation; bf16 in/out"
DTYPE_RMSNORM = "bf16 in/out, fp32 arithmetic"
DTYPE_NVFP4 = "packed FP4 (E2M1) x E4M3 1x16 block scales on the tcgen05 block-scaled MMA, fp32 accumulation, alpha folded; bf16 out"


def read_peaks():
    p = REPO / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured", d
    return FALLBACK_HBM_GBS, "fallback", {}


def kernel_hash(name: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[name]:
        h.update((REPO / "memory_bound_decode_fd_gb300" / rel).read_bytes())
    return h.hexdigest()[:12]


def recorded_traffic(name: str, tag: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel
    source (hash match); else None."""
    p = REPO / "profiles" / "traffic.md"
    if not p.exists():
        return None
    pat = re.compile(rf"^\|\s*{re.escape(name)}\s*\|\s*{re.escape(tag)}\s*\|\s*([0-9a-f]+)\s*\|\s*([0-9]+)\s*\|", re.M)
    m = pat.search(p.read_text())
    if not m or m.group(1) != kernel_hash(name):
        return None
    return int(m.group(2))


def smi_index() -> int:
    """nvidia-smi index of this rank's GPU (CUDA_VISIBLE_DEVICES remaps device ids)."""
    local = int(os.environ.get("LOCAL_RANK", 0))
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def time_region(stream, fn, iters: int) -> float:
    """ms for `iters` calls of fn on `stream`, CUDA events, synchronized on both sides."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(iters):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


# ----------------------------------------------------------------------------- workloads

def to_dev(bits_or_words, device):
    arr = np.ascontiguousarray(bits_or_words)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(arr).to(device)


def build_decode(device, seed=3, layers=32):
    import memory_bound_decode_fd_gb300 as fd
    from memory_bound_decode_fd_gb300 import inputs
    from memory_bound_decode_fd_gb300.step import DecodeStep

    spec = inputs.WORKLOADS["decode_step"]
    d = inputs.decode_step_inputs(layers=layers, hidden=spec["hidden"], inter=spec["inter"],
                                  group=spec["group"], seed=seed)
    dev_layers = [{"rms_weight": to_dev(L["rms_weight"], device),
                   "qweight": to_dev(L["qweight"], device),
                   "scales": to_dev(L["scales"], device)} for L in d["layers"]]
    step = DecodeStep(dev_layers, spec["hidden"], spec["inter"], spec["group"], spec["eps"], device)
    step.x.copy_(to_dev(d["x"], device))
    step.residual.copy_(to_dev(d["residual"], device))
    for i, L in enumerate(d["layers"]):
        step.gate[i].copy_(to_dev(L["gate"], device))
        step.up[i].copy_(to_dev(L["up"], device))
    step.capture()
    bytes_per_step = fd.decode_step_bytes(layers, spec["hidden"], spec["inter"], spec["group"])
    return d, step, bytes_per_step


DECODE_WORKLOAD = ("decode_step: 32 x [add-RMSNorm 1x4096 eps 1e-5 + SwiGLU-W4A16 GEMV M=1 "
                   "K=14336 N=4096 group 128], seed 3")


def decode_config(world: int) -> dict:
    """The decode-step workload's `config`, the same on the GPU arm and the reference arm."""
    from memory_bound_decode_fd_gb300 import traffic

    return {
        "workload": DECODE_WORKLOAD,
        "bytes_per_step": traffic.decode_step_bytes(32, 4096, 14336, 128),
        "l2": "inputs larger than L2 (972 MB of weights per step vs 129 MB L2); no flush",
        "parallelism": f"replicas x{world}",
    }


def bench_decode(args, device, rank, world):
    import memory_bound_decode_fd_gb300 as fd

    spec = {"layers": 32, "hidden": 4096, "inter": 14336, "group": 128, "eps": 1e-5}
    d, step, bytes_per_step = build_decode(device)
    stream = step.stream
    hbm_peak, peak_kind, peaks = read_peaks()

    sampler = ClockSampler(smi_index())
    sampler.start()
    # clocks settle + warm-up (untimed)
    settle_until = time.time() + 1.0
    while time.time() < settle_until:
        time_region(stream, step.replay, 200)
    time_region(stream, step.replay, max(args.warmup, 3))

    barrier(world)
    ms = time_region(stream, step.replay, args.steps)
    ms = max_over_ranks(ms, world)
    clocks = sampler.stop()
    ms_per_step = ms / args.steps
    value_gbs = job_throughput_gbs(world, bytes_per_step, ms_per_step)

    # Per-kernel durations: each kernel's launches of the step, captured alone in a CUDA
    # graph (same buffers and weights, programmatic dependent launch as in the step) and
    # replayed on the same stream; average launch duration = event time / launches.
    # Includes the small inter-kernel gap, so it is conservative. The step runs the 32
    # add-RMSNorm and 32 GEMV launches; the GEMV with the next layer's add-RMSNorm folded
    # in (fd_swiglu_w4a16_gemv_add_rmsnorm, not used by the step) is timed as well.
    hidden = spec["hidden"]
    L = spec["layers"]
    fold_scratch = fd.fold_scratch(device)
    kern_launch = {
        "swiglu_w4a16_gemv_add_rmsnorm": [lambda L_=ly, i=i: fd.swiglu_w4a16_gemv_add_rmsnorm(
            L_["gate"], L_["up"], L_["qweight"], L_["scales"], step.residual,
            step.layers[i + 1]["rms_weight"], spec["eps"], fold_scratch, y=step.y[i],
            normed=step.normed[i + 1], residual_out=step.residual, group=spec["group"], stream=stream)
            for i, ly in enumerate(step.layers[:-1])],
        "swiglu_w4a16_gemv": [lambda L_=ly, i=i: fd.swiglu_w4a16_gemv(
            L_["gate"], L_["up"], L_["qweight"], L_["scales"], out=step.y[i], group=spec["group"],
            stream=stream) for i, ly in enumerate(step.layers)],
        "add_rmsnorm": [lambda L_=ly, i=i: fd.add_rmsnorm(
            step.y[i - 1] if i else step.x, step.residual, L_["rms_weight"], spec["eps"],
            out=step.normed[i], residual_out=step.residual, stream=stream)
            for i, ly in enumerate(step.layers)],
    }
    kernels = {}
    prev_pdl = fd.set_pdl(step.pdl)
    try:
        for name, calls in kern_launch.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for c in calls:
                    c()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for c in calls:
                    c()
            reps = max(10, args.steps // 10)
            with torch.cuda.stream(stream):
                time_region(stream, g.replay, 3)
                ms_k = time_region(stream, g.replay, reps)
            kernels[name] = {"us": ms_k * 1e3 / (reps * len(calls)), "launches_timed": reps * len(calls)}
    finally:
        fd.set_pdl(prev_pdl)
    gemv_bytes = fd.gemv_bytes(1, spec["inter"], hidden, spec["group"])
    rms_bytes = fd.add_rmsnorm_bytes(1, hidden)
    # the folded call moves the GEMV's bytes plus the add-RMSNorm's minus its read of y,
    # which stays on chip: residual in, new residual and normalised row out, weight row
    fold_bytes = gemv_bytes + 8 * hidden
    kernels["swiglu_w4a16_gemv_add_rmsnorm"]["bytes"] = fold_bytes
    kernels["swiglu_w4a16_gemv"]["bytes"] = gemv_bytes
    kernels["add_rmsnorm"]["bytes"] = rms_bytes
    for k in kernels.values():
        k["gbs"] = k["bytes"] / (k["us"] * 1e-6) / 1e9
    gemv_us = kernels["swiglu_w4a16_gemv"]["us"]
    achieved = gemv_bytes / (gemv_us * 1e-6) / 1e9
    traffic = recorded_traffic("swiglu_w4a16_gemv", "K14336_N4096_M1")

    # The step launched eagerly (no CUDA graph: every launch pays the host's launch cost),
    # with separate kernels (64 launches) and with each later add-RMSNorm folded into the
    # GEMV before it (33 launches).
    eager = {}
    res_save = step.residual.clone()
    for name, sc in (("separate_64_launches", None), ("folded_33_launches", fold_scratch)):
        run = lambda sc=sc: fd.decode_mlp_step(step.x, step.residual, step.layers, spec["eps"],  # noqa: E731
                                               spec["group"], normed=step.normed, y=step.y,
                                               stream=stream, scratch=sc)
        with torch.cuda.stream(stream):
            time_region(stream, run, 3)
            n_eager = max(5, min(50, args.steps // 10))
            eager[name] = round(time_region(stream, run, n_eager) / n_eager, 4)
    step.residual.copy_(res_save)

    # End to end: pinned host inputs -> device, replay, device -> pinned host.
    pin = dict(dtype=torch.bfloat16, pin_memory=True)
    xh = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    rh = torch.from_numpy(d["residual"].view(np.int16)).view(torch.bfloat16).pin_memory()
    gh = torch.from_numpy(np.stack([L["gate"] for L in d["layers"]]).view(np.int16)).view(torch.bfloat16).pin_memory()
    uh = torch.from_numpy(np.stack([L["up"] for L in d["layers"]]).view(np.int16)).view(torch.bfloat16).pin_memory()
    ox = torch.empty((1, hidden), **pin)
    orr = torch.empty((1, hidden), **pin)
    e2e_call = lambda: step(xh, rh, gh, uh, ox, orr)  # noqa: E731
    time_region(stream, e2e_call, max(args.warmup, 3))
    barrier(world)
    e2e_sep_ms = max_over_ranks(time_region(stream, e2e_call, args.steps), world) / args.steps
    # the same through StepIO: one host->device copy of the step's inputs, one
    # device->host copy of its outputs
    io = step.pinned_io()
    io.x.copy_(xh)
    io.residual.copy_(rh)
    io.gate.copy_(gh)
    io.up.copy_(uh)
    step.capture_pinned(io)
    e2e_io = lambda: step.run_pinned(io)  # noqa: E731
    time_region(stream, e2e_io, max(args.warmup, 3))
    barrier(world)
    e2e_ms = max_over_ranks(time_region(stream, e2e_io, args.steps), world) / args.steps
    h2d = (xh.numel() + rh.numel() + gh.numel() + uh.numel()) * 2
    d2h = (ox.numel() + orr.numel()) * 2

    # The same step as one persistent cooperative launch (fd_decode_mlp_step: a memset and
    # one kernel per step, bit-identical outputs), captured in a graph and timed the same way.
    from memory_bound_decode_fd_gb300.step import DecodeStep
    pers = DecodeStep(step.layers, step.hidden, step.inter, step.group, step.eps, device,
                      persistent=True)
    pers.x.copy_(step.x)
    pers.residual.copy_(step.residual)
    pers.gate.copy_(step.gate)
    pers.up.copy_(step.up)
    pers.capture()
    with torch.cuda.stream(pers.stream):
        time_region(pers.stream, pers.replay, max(args.warmup, 3))
        barrier(world)
        pers_ms = max_over_ranks(time_region(pers.stream, pers.replay, args.steps), world) / args.steps
    persistent = {"ms_per_step": round(pers_ms, 6),
                  "value": round(job_throughput_gbs(world, bytes_per_step, pers_ms), 2),
                  "unit": "GB/s",
                  "launch": "fd_decode_mlp_step: one cooperative kernel (one CTA per SM, all 32 layers) and one memset per step"}
    del pers

    line = {
        "metric": METRIC,
        "value": round(value_gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_DP2A + "; add-RMSNorm " + DTYPE_RMSNORM,
        "data": "synthetic (seeded: int4 weights uniform on [-8,7], bf16 scales U[0.005,0.02], activations and residual N(0,1), norm weights N(1,0.1))",
        "config": decode_config(world),
        "launch": "one CUDA graph replay per step (64 kernels)",
        "pct_of_measured_hbm": round(100 * value_gbs / world / hbm_peak, 1),
        "pct_of_spec_8tbs": round(100 * value_gbs / world / SPEC_HBM_GBS, 1),
        "kernels": {k: {kk: (round(vv, 3) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                    for k, v in kernels.items()},
        "roofline": {
            "kernel": "swiglu_w4a16_gemv (M=1 K=14336 N=4096)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": hbm_peak,
            "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": gemv_bytes,
            "launches_per_step": L,
        },
        "e2e": {
            "value": round(job_throughput_gbs(world, bytes_per_step, e2e_ms), 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 6),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "api": "memory_bound_decode_fd_gb300.step.DecodeStep.run_pinned (StepIO captured with the step: fd_copy kernels read and write the pinned host block, one graph launch)",
            "four_copy_call_ms_per_step": round(e2e_sep_ms, 6),
        },
        "eager_ms_per_step": eager,
        "persistent_step": persistent,
        "gpu_launches": 2 * spec["layers"] * args.steps,
        "clocks": clocks,
    }
    if not args.no_configs:
        # Every other workload configuration, timed in this process (one call per step,
        # rotating input sets, CUDA graph with programmatic dependent launch).
        line["configs"] = {name: measure_workload(name, device, world, settle_s=0.3)
                           for name in CONFIG_WORKLOADS}
    return line, d


def cpu_baseline_decode(d, budget_s=12.0):
    """The oracle as it stands on this host's cores, on a bounded sample of the decode
    step: whole layers, in order, until `budget_s` of CPU time is spent."""
    import oracle
    from memory_bound_decode_fd_gb300 import traffic

    t0 = time.perf_counter()
    n = 0
    x, res = d["x"], d["residual"]
    for L in d["layers"]:
        rec, x, res = oracle.decode_mlp_step(x, res, [L], 1e-5, d["group"])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    b = n * (traffic.add_rmsnorm_bytes(1, d["hidden"]) + traffic.gemv_bytes(1, d["inter"], d["hidden"], d["group"]))
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} of 32 decode-step layers (add-RMSNorm 1x4096 + GEMV 14336x4096 each), {dt:.1f} s, float64 numpy, 1 thread"}


def oracle_sampler(workload: str):
    """A bounded sample of `workload` for the CPU oracle: returns (run(i, rows), bytes(rows),
    total rows, description). One sample is the workload's call restricted to `rows` of
    its output rows (weight rows of a GEMV, rows of an add-RMSNorm); the decode step's
    sample is one layer's add-RMSNorm plus that layer's GEMV over `rows` output rows."""
    import oracle
    from memory_bound_decode_fd_gb300 import inputs, traffic

    spec = dict(inputs.WORKLOADS[workload])
    kind = spec.pop("kind")
    if kind == "decode":
        d = inputs.decode_step_inputs(layers=32, seed=spec["seed"])
        hidden, inter, group = d["hidden"], d["inter"], d["group"]

        def run(i, rows):
            L = d["layers"][i % 32]
            lo = (i * 97) % (hidden - rows + 1)
            oracle.add_rmsnorm(d["x"], d["residual"], L["rms_weight"], spec["eps"])
            oracle.swiglu_w4a16_gemv(L["gate"], L["up"], L["qweight"][lo:lo + rows],
                                     L["scales"][lo:lo + rows], group)

        nbytes = lambda rows: traffic.add_rmsnorm_bytes(1, hidden) + traffic.gemv_bytes(1, inter, rows, group)  # noqa: E731
        return run, nbytes, hidden, "one layer's add-RMSNorm 1x4096 + its GEMV over {rows} of 4096 output rows"
    if kind in ("gemv", "batched", "gemv_residual"):
        M, K, N, g = spec["M"], spec["K"], spec["N"], spec["group"]
        d = inputs.gemv_inputs(M, K, N, g, seed=spec["seed"])
        res = inputs.normal_bf16(np.random.default_rng(spec["seed"] + 1), (M, N))

        def run(i, rows):
            lo = (i * 97) % (N - rows + 1)
            if kind == "gemv_residual":
                oracle.swiglu_w4a16_gemv_residual(d["gate"], d["up"], d["qweight"][lo:lo + rows],
                                                  d["scales"][lo:lo + rows],
                                                  np.ascontiguousarray(res[:, lo:lo + rows]), g)
            else:
                oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"][lo:lo + rows],
                                         d["scales"][lo:lo + rows], g)

        extra = (lambda rows: M * rows * 2) if kind == "gemv_residual" else (lambda rows: 0)
        nbytes = lambda rows: traffic.gemv_bytes(M, K, rows, g) + extra(rows)  # noqa: E731
        return run, nbytes, N, f"GEMV M={M} K={K} over {{rows}} of {N} output rows"
    if kind == "gate_up":
        M, K, inter, g = spec["M"], spec["K"], spec["I"], spec["group"]
        rng = np.random.default_rng(spec["seed"])
        x = inputs.normal_bf16(rng, (M, K))
        q = inputs.int4_words(rng, 2 * inter, K)
        sc = inputs.scales_bf16(rng, 2 * inter, K, g)

        def run(i, rows):
            lo = (i * 97) % (2 * inter - rows + 1)
            oracle.w4a16_gemv(x, q[lo:lo + rows], sc[lo:lo + rows], g)

        nbytes = lambda rows: rows * K // 2 + rows * (K // g) * 2 + M * K * 2 + M * rows * 2  # noqa: E731
        return run, nbytes, 2 * inter, f"gate/up GEMV M={M} K={K} over {{rows}} of {2 * inter} stacked rows"
    if kind == "nvfp4":
        M, K, N = spec["M"], spec["K"], spec["N"]
        d = inputs.nvfp4_inputs(M, K, N, seed=spec["seed"])

        def run(i, rows):
            lo = (i * 97) % (N - rows + 1)
            oracle.nvfp4_scaled_mm(d["x"], d["x_sf"], d["w"][lo:lo + rows], d["w_sf"][lo:lo + rows], d["alpha"])

        nbytes = lambda rows: traffic.nvfp4_bytes(M, K, rows)  # noqa: E731
        return run, nbytes, N, f"NVFP4 scaled matmul M={M} K={K} over {{rows}} of {N} weight rows"
    rows_all, hidden = spec["rows"], spec["hidden"]
    d = inputs.rmsnorm_inputs(rows_all, hidden, seed=spec["seed"])

    def run(i, rows):
        lo = (i * 97) % (rows_all - rows + 1)
        oracle.add_rmsnorm(d["x"][lo:lo + rows], d["residual"][lo:lo + rows], d["weight"], spec["eps"])

    nbytes = lambda rows: traffic.add_rmsnorm_bytes(rows, hidden)  # noqa: E731
    return run, nbytes, rows_all, f"add-RMSNorm over {{rows}} of {rows_all} rows x {hidden}"


def reference_arm(args):
    """`--impl reference`: the CPU oracle, as it stands, timed on the host cores (one
    thread). Each step is a bounded sample of the workload (see oracle_sampler), sized so
    that the whole --steps K --warmup W run ends within a few minutes; ms_per_step is
    the measured time of one sample."""
    run, nbytes, total_rows, what = oracle_sampler(args.workload)
    total = args.steps + args.warmup
    target_s = min(2.0, max(0.02, 150.0 / max(total, 1)))

    def sample(i, rows):
        t0 = time.perf_counter()
        run(i, rows)
        return time.perf_counter() - t0

    # calibrate the slice so one sample takes about target_s (re-measured, since a sample
    # has fixed costs besides its per-row work)
    rows = min(64, total_rows)
    for _ in range(4):
        t = sample(0, rows)
        new_rows = int(max(min(8, total_rows), min(total_rows, rows * target_s / max(t, 1e-6))))
        if abs(new_rows - rows) <= 0.25 * rows:
            break
        rows = new_rows
    sample_bytes = nbytes(rows)
    times = []
    for i in range(total):
        dt = sample(i, rows)
        if i >= args.warmup:
            times.append(dt)
    if not times:
        times.append(sample(0, rows))
    per = sum(times) / len(times)
    value = sample_bytes / per / 1e9
    desc = what.format(rows=rows)
    if args.workload == "decode_step":
        config = decode_config(1)
        full_bytes = config["bytes_per_step"]
    else:
        config = {"workload": args.workload, "parallelism": "replicas x1"}
        full_bytes = None
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": config,
        "sample": f"per step: {desc} ({sample_bytes} B), float64 numpy oracle, 1 thread",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(times)} samples of {desc}, float64 numpy, 1 thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if full_bytes:
        # the whole 32-layer step at the sample's rate (an extrapolation, not a measurement)
        line["ms_per_full_step_extrapolated"] = round(full_bytes / (value * 1e9) * 1e3, 3)
    return line


# ----------------------------------------------------------------------------- single-call workloads

# The workload configurations measured in the default run's "configs" object, besides the
# decode step itself: the small GEMV, the 8192 x 4096 add-RMSNorm and the K=9216 N=2560
# GEMV (the two shapes held to the 70 % target), the batched M=64 product (tensor-core
# vs CUDA-core kernel), the fused layer's other two kernels and the NVFP4 QKV projection.
CONFIG_WORKLOADS = ["gemv_small", "rmsnorm_big", "gemv_94mb", "batched_m64", "gemv_residual", "gate_up",
                    "nvfp4_qkv"]
TARGET_PCT = {"rmsnorm_big": 70.0, "gemv_94mb": 70.0}


def build_single_calls(name, device, l2):
    """The calls of one single-call workload: every call reads a different input set
    (ceil(3 x L2 / bytes) sets) so that each reads HBM. Returns (calls, nbytes, kernel
    name, description, extra) where extra holds the shape for the path comparison."""
    import memory_bound_decode_fd_gb300 as fd
    from memory_bound_decode_fd_gb300 import inputs

    spec = dict(inputs.WORKLOADS[name])
    kind = spec.pop("kind")
    calls = []
    extra = {"kind": kind}
    if kind in ("gemv", "batched", "gemv_residual"):
        M, K, N, g = spec["M"], spec["K"], spec["N"], spec["group"]
        extra.update(M=M, K=K, N=N, group=g)
        if fd.gemv_uses_tensor_cores(M, K, N, g):
            extra.update(traffic_kernel="gemv_tc", traffic_tag=f"M{M}_K{K}_N{N}")
        else:
            extra["traffic_tag"] = f"K{K}_N{N}_M{M}"
        with_res = kind == "gemv_residual"
        nbytes = fd.gemv_bytes(M, K, N, g) + (M * N * 2 if with_res else 0)
        nsets = max(1, min(4096, math.ceil(3 * l2 / nbytes)))
        base = inputs.gemv_inputs(M, K, N, g, seed=spec["seed"])
        gate, up = to_dev(base["gate"], device), to_dev(base["up"], device)
        rng = np.random.default_rng(spec["seed"] + 1)
        qs = [to_dev(base["qweight"], device)] + [to_dev(inputs.int4_words(rng, N, K), device) for _ in range(nsets - 1)]
        ss = [to_dev(base["scales"], device)] + [to_dev(inputs.scales_bf16(rng, N, K, g), device) for _ in range(nsets - 1)]
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        if with_res:
            # the residual stream x (read) and the new residual (written to `out`)
            res = to_dev(inputs.normal_bf16(rng, (M, N)), device)
            for q, s_ in zip(qs, ss):
                calls.append(lambda q=q, s_=s_: fd.swiglu_w4a16_gemv_residual(gate, up, q, s_, res, out=out, group=g))
            kname = "swiglu_w4a16_gemv_residual"
            desc = f"GEMV + residual-add epilogue M={M} K={K} N={N} group {g}, seed {spec['seed']}"
        else:
            for q, s_ in zip(qs, ss):
                calls.append(lambda q=q, s_=s_: fd.swiglu_w4a16_gemv(gate, up, q, s_, out=out, group=g))
            kname, desc = "swiglu_w4a16_gemv", f"GEMV M={M} K={K} N={N} group {g}, seed {spec['seed']}"
    elif kind == "gate_up":
        M, K, inter, g = spec["M"], spec["K"], spec["I"], spec["group"]
        # stacked int4 weights [2I, K] and scales, x once, g and u written
        nbytes = fd.gate_up_bytes(M, K, inter, g)
        nsets = max(1, min(4096, math.ceil(3 * l2 / nbytes)))
        rng = np.random.default_rng(spec["seed"])
        x = to_dev(inputs.normal_bf16(rng, (M, K)), device)
        gout = torch.empty((M, inter), dtype=torch.bfloat16, device=device)
        uout = torch.empty_like(gout)
        for _ in range(nsets):
            q = to_dev(inputs.int4_words(rng, 2 * inter, K), device)
            s_ = to_dev(inputs.scales_bf16(rng, 2 * inter, K, g), device)
            calls.append(lambda q=q, s_=s_: fd.w4a16_gate_up_gemv(x, q, s_, gate_out=gout, up_out=uout, group=g))
        kname = "w4a16_gate_up_gemv"
        extra["traffic_tag"] = f"K{K}_I{inter}_M{M}"
        desc = f"gate/up GEMV (horizontal fusion) M={M} K={K} I={inter} (2I={2 * inter} rows) group {g}, seed {spec['seed']}"
    elif kind == "nvfp4":
        M, K, N = spec["M"], spec["K"], spec["N"]
        extra.update(M=M, K=K, N=N)
        nbytes = fd.nvfp4_bytes(M, K, N)
        nsets = max(1, min(4096, math.ceil(3 * l2 / nbytes)))
        d = inputs.nvfp4_inputs(M, K, N, seed=spec["seed"])
        x, xs = to_dev(d["x"], device), to_dev(d["x_sf"], device)
        alpha = torch.tensor([float(d["alpha"])], dtype=torch.float32, device=device)
        rng = np.random.default_rng(spec["seed"] + 1)
        ws = [(to_dev(d["w"], device), to_dev(d["w_sf"], device))] + [
            (to_dev(inputs.fp4_bytes(rng, N, K), device), to_dev(inputs.e4m3_scale_codes(rng, N, K), device))
            for _ in range(nsets - 1)]
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        for w, wsf in ws:
            calls.append(lambda w=w, wsf=wsf: fd.nvfp4_scaled_mm(x, xs, w, wsf, alpha, out=out))
        kname = "nvfp4_scaled_mm"
        extra["traffic_tag"] = f"M{M}_K{K}_N{N}"
        desc = (f"NVFP4 scaled matmul, output multiplier folded in, M={M} K={K} N={N} "
                f"(E2M1, E4M3 1x16 block scales), seed {spec['seed']}")
    else:
        rows, hidden = spec["rows"], spec["hidden"]
        nbytes = fd.add_rmsnorm_bytes(rows, hidden)
        nsets = max(1, min(64, math.ceil(3 * l2 / nbytes)))
        d = inputs.rmsnorm_inputs(rows, hidden, seed=spec["seed"])
        w = to_dev(d["weight"], device)
        sets = [(to_dev(d["x"], device), to_dev(d["residual"], device)) for _ in range(nsets)]
        y = torch.empty((rows, hidden), dtype=torch.bfloat16, device=device)
        h = torch.empty_like(y)
        for x, r in sets:
            calls.append(lambda x=x, r=r: fd.add_rmsnorm(x, r, w, spec["eps"], out=y, residual_out=h))
        kname, desc = "add_rmsnorm", f"add-RMSNorm rows={rows} hidden={hidden} eps {spec['eps']}, seed {spec['seed']}"
        extra["traffic_tag"] = f"R{rows}_H{hidden}"
    return calls, nbytes, kname, desc, extra


def capture_calls(calls, stream):
    """The calls as one CUDA graph, launched back to back as a decode engine issues them:
    programmatic dependent launch between consecutive kernels (each still waits for its
    predecessor before it reads activations or writes outputs; results are bitwise those
    of plain launches)."""
    import memory_bound_decode_fd_gb300 as fd

    prev_pdl = fd.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            for c in calls:
                c()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for c in calls:
                c()
    finally:
        fd.set_pdl(prev_pdl)
    return gr


def measure_workload(name, device, world, steps=None, warmup=3, target_ms=300.0, settle_s=1.0):
    """Times one single-call workload. With `steps` the timed region holds at least that
    many calls; otherwise enough graph replays to fill about `target_ms`. Returns a dict
    with the per-call time, GB/s and the fraction of the measured HBM bandwidth."""
    import memory_bound_decode_fd_gb300 as fd

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    calls, nbytes, kname, desc, extra = build_single_calls(name, device, l2)
    kind = extra["kind"]
    stream = torch.cuda.Stream(device)
    graph = capture_calls(calls, stream)
    replay = graph.replay
    with torch.cuda.stream(stream):
        time_region(stream, replay, 1)
        t_one = max(time_region(stream, replay, 1), 1e-3)
    if steps is not None:
        reps = max(1, math.ceil(steps / len(calls)))
    else:
        reps = max(3, math.ceil(target_ms / t_one))
    compare = None
    if kind == "batched":
        # The batched shape runs on the tensor-core kernel; time the CUDA-core kernel on
        # the same calls for comparison (a short run: it is compute bound).
        M, K, N, g = extra["M"], extra["K"], extra["N"], extra["group"]
        compare = {"selected": "tensor" if fd.gemv_uses_tensor_cores(M, K, N, g) else "cuda_core"}
        for path in ("tensor", "cuda_core"):
            prev = fd.set_gemv_path(path)
            try:
                gr = capture_calls(calls, stream)
            finally:
                fd.set_gemv_path(prev)
            with torch.cuda.stream(stream):
                time_region(stream, gr.replay, 2)
                n = 2 if path == "cuda_core" else max(2, reps // 4)
                t_ms = time_region(stream, gr.replay, n)
            us = t_ms * 1e3 / (n * len(calls))
            compare[f"{path}_us_per_call"] = round(us, 3)
            compare[f"{path}_tflops"] = round(fd.gemv_flops(M, K, N) / (us * 1e-6) / 1e12, 1)
            compare[f"{path}_gbs"] = round(nbytes / (us * 1e-6) / 1e9, 1)
            del gr
    hbm_peak, _, _ = read_peaks()
    sampler = ClockSampler(smi_index())
    sampler.start()
    settle_until = time.time() + settle_s
    with torch.cuda.stream(stream):
        while time.time() < settle_until:
            time_region(stream, replay, 10)
        time_region(stream, replay, max(warmup, 3))
        barrier(world)
        ms = max_over_ranks(time_region(stream, replay, reps), world)
    clocks = sampler.stop()
    n_calls = reps * len(calls)
    us_call = ms * 1e3 / n_calls
    gbs = nbytes / (us_call * 1e-6) / 1e9
    if kind == "nvfp4":
        dtype = DTYPE_NVFP4
    elif "gemv" not in kname:
        dtype = DTYPE_RMSNORM
    elif kind in ("gemv", "batched", "gemv_residual") and fd.gemv_uses_tensor_cores(
            extra["M"], extra["K"], extra["N"], extra["group"]):
        dtype = DTYPE_TC
    else:
        dtype = DTYPE_DP2A
    rec = {
        "workload": f"{name}: {desc}",
        "kernel": kname,
        "bytes_per_call": nbytes,
        "us_per_call": round(us_call, 3),
        "gbs": round(gbs, 1),
        "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
        "pct_of_measured_hbm": round(100 * gbs / hbm_peak, 1),
        "pct_of_spec_8tbs": round(100 * gbs / SPEC_HBM_GBS, 1),
        "calls_timed": n_calls,
        "input_sets": len(calls),
        "dtype": dtype,
        "clocks": clocks,
    }
    if name in TARGET_PCT:
        rec["target_pct_of_peak"] = TARGET_PCT[name]
        rec["meets_target"] = bool(rec["pct_of_measured_hbm"] >= TARGET_PCT[name])
    if kind == "nvfp4":
        rec["tflops"] = round(fd.nvfp4_flops(extra["M"], extra["K"], extra["N"]) / (us_call * 1e-6) / 1e12, 1)
    if compare:
        rec["paths"] = compare
    if extra.get("traffic_tag"):
        rec["traffic"] = recorded_traffic(extra.get("traffic_kernel", kname), extra["traffic_tag"])
    return rec


def bench_single(args, device, rank, world):
    rec = measure_workload(args.workload, device, world, steps=args.steps, warmup=args.warmup)
    hbm_peak, peak_kind, _ = read_peaks()
    us_call = rec["us_per_call"]
    gbs_job = world * rec["gbs"]
    return {
        "metric": METRIC, "value": round(gbs_job, 2), "unit": "GB/s", "n_gpus": world,
        "steps": rec["calls_timed"], "warmup": args.warmup, "ms_per_step": round(us_call / 1e3, 6),
        "us_per_call": us_call, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": rec["dtype"],
        "data": "synthetic (seeded)",
        "config": {"workload": rec["workload"], "bytes_per_call": rec["bytes_per_call"],
                   "l2": f"{rec['input_sets']} rotating input sets ({rec['input_sets']} x {rec['bytes_per_call']} B vs L2)",
                   "parallelism": f"replicas x{world}"},
        "launch": f"CUDA graph of {rec['input_sets']} calls, programmatic dependent launch",
        "pct_of_measured_hbm": rec["pct_of_measured_hbm"],
        "pct_of_spec_8tbs": rec["pct_of_spec_8tbs"],
        "roofline": {"kernel": rec["kernel"], "bound": "hbm", "achieved": rec["gbs"],
                     "peak": hbm_peak, "unit": "GB/s", "frac": rec["frac_of_measured_hbm"],
                     "kernel_us": us_call, "traffic": rec.get("traffic")},
        "e2e": None,
        "gpu_launches": rec["calls_timed"],
        "clocks": rec["clocks"],
        **({"paths": rec["paths"]} if "paths" in rec else {}),
    }


def bench_fused_layer(args, device, rank, world):
    """32 decode layers of the pages' fully fused form, one CUDA graph with programmatic
    dependent launch: add_rmsnorm(x, h) -> (normed, h); g, u = gate_up(normed);
    h = h + down(silu(g) * u) in place. Llama-3-8B shapes (hidden 4096, MLP 14336). The
    2.9 GB of int4 weights are drawn on the device (seeded); x_next of a layer is the
    normed row of the next (x is the same tensor), so the step is one residual stream."""
    import memory_bound_decode_fd_gb300 as fd

    L, hidden, inter, g, eps, seed = 32, 4096, 14336, 128, 1e-5, 3
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def words(n, k):
        return torch.randint(-2**31, 2**31 - 1, (n, k // 8), generator=gen, device=device, dtype=torch.int32)

    def scales(n, k):
        return (0.005 + 0.015 * torch.rand((n, k // g), generator=gen, device=device)).to(torch.bfloat16)

    layers = [dict(w=(1.0 + 0.1 * torch.randn(hidden, generator=gen, device=device)).to(torch.bfloat16),
                   qgu=words(2 * inter, hidden), sgu=scales(2 * inter, hidden),
                   qd=words(hidden, inter), sd=scales(hidden, inter)) for _ in range(L)]
    x = torch.randn((1, hidden), generator=gen, device=device).to(torch.bfloat16)
    h = torch.randn((1, hidden), generator=gen, device=device).to(torch.bfloat16)
    normed = torch.empty_like(x)
    gt = torch.empty((1, inter), dtype=torch.bfloat16, device=device)
    ut = torch.empty_like(gt)
    zero = torch.zeros_like(x)

    def step():
        for i, ly in enumerate(layers):
            # layer 0 adds the incoming x; later layers' residual stream is h alone
            fd.add_rmsnorm(x if i == 0 else zero, h, ly["w"], eps, out=normed, residual_out=h)
            fd.w4a16_gate_up_gemv(normed, ly["qgu"], ly["sgu"], gate_out=gt, up_out=ut, group=g)
            fd.swiglu_w4a16_gemv_residual(gt, ut, ly["qd"], ly["sd"], h, out=h, group=g)

    stream = torch.cuda.Stream(device)
    prev = fd.set_pdl(True)
    try:
        stream.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    finally:
        fd.set_pdl(prev)
    per_layer = (fd.add_rmsnorm_bytes(1, hidden) + fd.gate_up_bytes(1, hidden, inter, g)
                 + fd.gemv_bytes(1, inter, hidden, g) + hidden * 2)
    nbytes = L * per_layer
    hbm_peak, peak_kind, _ = read_peaks()
    sampler = ClockSampler(smi_index())
    sampler.start()
    with torch.cuda.stream(stream):
        time_region(stream, graph.replay, max(args.warmup, 3))
        barrier(world)
        ms = max_over_ranks(time_region(stream, graph.replay, args.steps), world)
    clocks = sampler.stop()
    ms_step = ms / args.steps
    gbs = job_throughput_gbs(world, nbytes, ms_step)
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "us_per_step": round(ms_step * 1e3, 3), "us_per_layer": round(ms_step * 1e3 / L, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_DP2A + "; add-RMSNorm " + DTYPE_RMSNORM, "data": "synthetic (seeded, drawn on the device)",
        "config": {"workload": f"fused_layer: {L} x [add-RMSNorm 1x{hidden} + gate/up GEMV K={hidden} I={inter} "
                               f"+ down GEMV K={inter} N={hidden} with SwiGLU prologue and residual epilogue], seed {seed}",
                   "bytes_per_step": nbytes, "l2": f"{nbytes} B of weights per step vs L2 (defeats it)",
                   "launch": f"one CUDA graph of {3 * L} launches, programmatic dependent launch"},
        "pct_of_measured_hbm": round(100 * gbs / world / hbm_peak, 1),
        "roofline": None, "e2e": None, "gpu_launches": 3 * L * args.steps, "clocks": clocks,
    }


# ----------------------------------------------------------------------------- distributed plumbing

def bench_persistent(args, device, rank, world):
    """The decode step (add-RMSNorm + SwiGLU-W4A16 GEMV per layer, Llama-3-8B shapes) as one
    persistent cooperative launch, fd_decode_mlp_step: one CTA per SM for all layers, the
    outputs bit-identical to the chain of separate kernels. Timed as a CUDA graph of the
    memset and the kernel; end to end through DecodeStep.run_pinned."""
    import memory_bound_decode_fd_gb300 as fd
    from memory_bound_decode_fd_gb300.step import DecodeStep

    L = args.layers
    d, base, bytes_per_step = build_decode(device, layers=L)
    step = DecodeStep(base.layers, base.hidden, base.inter, base.group, base.eps, device,
                      persistent=True)
    step.x.copy_(base.x)
    step.residual.copy_(base.residual)
    step.gate.copy_(base.gate)
    step.up.copy_(base.up)
    step.capture()
    del base
    stream = step.stream
    hbm_peak, peak_kind, _ = read_peaks()
    sampler = ClockSampler(smi_index())
    sampler.start()
    with torch.cuda.stream(stream):
        time_region(stream, step.replay, max(args.warmup, 3))
        barrier(world)
        ms = max_over_ranks(time_region(stream, step.replay, args.steps), world) / args.steps
    clocks = sampler.stop()
    io = step.pinned_io()
    io.x.copy_(step.x.cpu())
    io.residual.copy_(step.residual.cpu())
    io.gate.copy_(step.gate.cpu())
    io.up.copy_(step.up.cpu())
    step.capture_pinned(io)
    with torch.cuda.stream(stream):
        time_region(stream, lambda: step.run_pinned(io), max(args.warmup, 3))
        barrier(world)
        e2e_ms = max_over_ranks(time_region(stream, lambda: step.run_pinned(io), args.steps), world) / args.steps
    h2d, d2h = io.h2d_bytes, io.d2h_bytes
    gbs = job_throughput_gbs(world, bytes_per_step, ms)
    # DRAM bytes per launch: the 8-layer ncu capture, scaled by the layers (every layer
    # moves the same bytes)
    t8 = recorded_traffic("decode_step", "L8")
    traffic = None if t8 is None else int(round(t8 * L / 8))
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_DP2A + "; add-RMSNorm " + DTYPE_RMSNORM,
        "data": "synthetic (seeded, as the decode_step workload)",
        "config": {"workload": f"persistent_step: {L} x [add-RMSNorm 1x4096 eps 1e-5 + SwiGLU-W4A16 "
                               "GEMV M=1 K=14336 N=4096 group 128], seed 3, one cooperative launch",
                   "bytes_per_step": bytes_per_step,
                   "l2": f"inputs larger than L2 ({bytes_per_step / 1e6:.0f} MB per step vs 129 MB L2); no flush",
                   "parallelism": f"replicas x{world}"},
        "launch": "CUDA graph of one memset and one cooperative kernel per step",
        "pct_of_measured_hbm": round(100 * gbs / world / hbm_peak, 1),
        "roofline": {"kernel": "decode_step_kernel (the whole step)", "bound": "hbm",
                     "achieved": round(gbs / world, 1), "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(gbs / world / hbm_peak, 4), "traffic": traffic,
                     "traffic_note": "8-layer capture scaled by layers / 8"},
        "e2e": {"value": round(job_throughput_gbs(world, bytes_per_step, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 6), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "memory_bound_decode_fd_gb300.step.DecodeStep(persistent=True).run_pinned"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time: every rank gets the maximum of `value` over all ranks."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s of N independent replicas: every rank moves `bytes_per_step` per
    step, and the job's step time is the slowest rank's (max over ranks)."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--workload", default="decode_step",
                    choices=["decode_step", "gemv_94mb", "rmsnorm_big", "gemv_small", "batched_m64",
                             "gemv_residual", "gate_up", "nvfp4_qkv", "fused_layer",
                             "persistent_step"])
    ap.add_argument("--layers", type=int, default=32, help="persistent_step: layers per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="decode step only: skip timing the other workload configurations")
    args = ap.parse_args(argv)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        if rank == 0:
            if args.workload == "fused_layer":
                line = {"impl": "reference", "unavailable": "the oracle has no gate/up-fed fused-layer chain; "
                        "its parts are timed by --workload gate_up and gemv_residual"}
            elif args.workload == "persistent_step":
                line = {"impl": "reference", "unavailable": "the same computation as decode_step "
                        "(bit-identical outputs): --workload decode_step times the oracle on it"}
            else:
                line = reference_arm(args)
            print(json.dumps(line), flush=True)
        return 0

    from memory_bound_decode_fd_gb300 import build

    build.build()  # no-op when libfd.so is up to date
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    if args.workload == "decode_step":
        line, d = bench_decode(args, device, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_decode(d)
    elif args.workload == "fused_layer":
        line = bench_fused_layer(args, device, rank, world)
    elif args.workload == "persistent_step":
        line = bench_persistent(args, device, rank, world)
    else:
        line = bench_single(args, device, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
