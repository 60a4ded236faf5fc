#!/usr/bin/env python
"""bench.py -- DDPM core fused forward+backward throughput on one GB300.

One step = one ddpm_forward plus one ddpm_backward (fused generator + dynamic
dilated depthwise filter, then dX / dY / dW / dbias with recomputed taps) over
one batch of the synthetic workload B=1, C=64, K=3, 256x256, bf16, inputs
resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU FP64 oracle (the plain C restatement of the
method under oracle/) on the host cores, on a bounded sample of the same
workload: the operator has no other runnable reference here.

Timing: CUDA events on the launching stream around each step, a 256 MiB
write between steps flushes the 129 MB L2 (outside the events), W untimed
warm-up steps, barrier + synchronize on both sides, max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DDPM fused fwd+bwd Mpixel/s (C=64,K=3,256² bf16, 1 GB300); % of roofline"
# metric names of the other steps (--step forward / filter), same unit
STEP_METRIC = {"train": METRIC,
               "forward": "DDPM fused generator+filter forward Mpixel/s (1 GB300); % of roofline",
               "filter": "DDPM filter with pregenerated taps Mpixel/s (1 GB300); % of HBM roofline",
               "filter_train": "DDPM filter with pregenerated taps fwd+bwd Mpixel/s (1 GB300); % of HBM roofline"}
UNIT = "Mpixel/s"
DEFAULT_WORKLOAD = "b1_c64_256x256_k3"
FLUSH_BYTES = 256 << 20

# Nominal GB300 unit counts used for the CUDA-core (FFMA) ceiling.
NUM_SMS = 152
FP32_LANES_PER_SM = 128
# Nominal dense tensor rates (PFLOP/s): a TF32 contraction is measured against the
# measured bf16 peak times their ratio.
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25


def load_peaks():
    """Measured HBM / bf16 peaks (driver-written), else the stated fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "sm_max_mhz": float(m.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


def fp32_alu_tflops(peaks) -> float:
    """FFMA ceiling: SMs x FP32 lanes x 2 flops x max SM clock."""
    return NUM_SMS * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


def kernel_work(name: str, p, es: int, splits: int):
    """Algorithmic work of one launch of a kernel: (bound, amount, unit-kind).

    flops count the contractions the kernel performs (2 per multiply-add);
    bytes count each input read once and each output written once.
    """
    P = p.B * p.H * p.W
    O = p.O
    C = p.C
    gemm = 2.0 * O * C * P
    if name == "filter_pregenerated_simt":
        return "hbm", P * (O + C + 4 * C) * es, "bytes"
    if name == "filter_bwd_dx":            # reads the taps and grad (4C), writes dx
        return "hbm", P * (O + 4 * C + C) * es, "bytes"
    if name == "filter_bwd_dtaps":         # reads grad blocks 1..3 and x, writes dtaps
        return "hbm", P * (3 * C + C + O) * es, "bytes"
    if name in ("forward_simt", "bwd_dx_simt", "bwd_dy_simt"):
        return "alu", gemm, "flops"
    if name == "bwd_dw_partial_simt":
        return "alu", 2.0 * O * (C + 1) * P, "flops"
    if name == "bwd_dw_reduce":
        return "hbm", splits * O * (C + 1) * 4 + O * (C + 1) * es, "bytes"
    if name == "pack_chunks":
        return "hbm", 2 * P * 4 * C * es, "bytes"
    if name == "pack_f32":                 # y and grad blocks 1..3 read, their channel-chunked copies written
        return "hbm", 2 * P * 4 * C * es, "bytes"
    if name in ("forward_tc", "bwd_dx_tc", "bwd_dx_tc_packed", "bwd_dx_gather", "bwd_dy_tc", "bwd_dw_tc"):
        return "tensor", gemm, "flops"
    if name == "bwd_dw_tf32":
        return "tensor_tf32", 2.0 * O * (C + 1) * P, "flops"
    if name == "forward_tf32":             # the algorithm's contraction (the kernel issues it as 3 TF32 products)
        return "tensor_tf32", gemm, "flops"
    if name in ("bwd_dy_tf32", "bwd_dx_tf32"):
        return "tensor_tf32", gemm, "flops"
    return "unknown", 0.0, "flops"


def step_roofline_us(p, es: int, peaks, step: str = "train") -> dict:
    """Roofline of one step: max(GEMM flops at the bf16 tensor peak, minimum
    bytes at the HBM peak).
      train   (fwd+bwd): four contractions of 2*O*C flops per pixel (generator,
              generator recompute for dX, dY, dW); x, y, weight, bias and grad
              read once, out / dx / dy / dW / dbias written once;
      forward: one contraction; x, y, weight, bias read, out written;
      filter:  no contraction; x and the taps read, out written;
      filter_train: no contraction; x, the taps and grad read, out, dx and dtaps written."""
    P = p.B * p.H * p.W
    w_bytes = (p.O * p.C + p.O) * es
    if step == "train":
        flops = 4 * 2.0 * p.O * p.C * P
        nbytes = P * (2 * p.C + 4 * p.C) * es + P * (4 * p.C + 2 * p.C + 2 * p.C) * es + 4 * w_bytes
    elif step == "forward":
        flops = 2.0 * p.O * p.C * P
        nbytes = P * (2 * p.C + 4 * p.C) * es + w_bytes
    elif step == "filter_train":
        flops = 0.0
        nbytes = P * (p.C + p.O + 4 * p.C + 4 * p.C + p.C + p.O) * es
    else:
        flops = 0.0
        nbytes = P * (p.C + p.O + 4 * p.C) * es
    t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    return {"flops": flops, "bytes": nbytes, "tensor_us": t_tc, "hbm_us": t_hbm, "roofline_us": max(t_tc, t_hbm)}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.out = os.path.join("/tmp", f"ddpm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out) as f:
            for line in f:
                cols = [c.strip() for c in line.split(",")]
                if len(cols) < 9:
                    continue
                try:
                    sm.append(float(cols[1]))
                    smax.append(float(cols[2]))
                except ValueError:
                    continue
                for n, v in zip(names, cols[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.out)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# The source file of each kernel whose ncu traffic is stored (all of them also
# depend on every shared header, .cuh / .h).
KERNEL_SOURCE = {"forward_tc": "forward_tc.cu", "pack_chunks": "bwd_dx_packed.cu",
                 "bwd_dx_tc_packed": "bwd_dx_packed.cu", "bwd_dy_tc": "bwd_dy_tc.cu", "bwd_dw_tc": "bwd_dw_tc.cu",
                 "bwd_dw_reduce": "backward_simt.cu", "bwd_dx_tc": "bwd_dx_tc.cu", "bwd_dw_tf32": "bwd_dw_tf32.cu",
                 "forward_tf32": "forward_tf32.cu", "forward_simt": "forward_simt.cu",
                 "filter_pregenerated_simt": "filter_simt.cu", "filter_bwd_dx": "filter_bwd_simt.cu",
                 "filter_bwd_dtaps": "filter_bwd_simt.cu", "bwd_dx_simt": "backward_simt.cu",
                 "bwd_dy_simt": "backward_simt.cu", "bwd_dw_partial_simt": "backward_simt.cu",
                 "bwd_dy_tf32": "bwd_dy_tf32.cu", "bwd_dx_tf32": "bwd_dx_tf32.cu", "pack_f32": "bwd_dx_tf32.cu",
                 "bwd_dx_gather": "bwd_dx_gather.cu"}


def kernel_source_digest(kernel: str) -> str:
    """Digest of a kernel's source file and of every shared header (to invalidate
    its stored ncu traffic figure once any of them changes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dynamic_dilated_depthwise_gb300", "csrc")
    names = sorted(n for n in os.listdir(csrc) if n.endswith((".cuh", ".h")))
    names.append(KERNEL_SOURCE.get(kernel, ""))
    for name in names:
        path = os.path.join(csrc, name)
        if not os.path.isfile(path):
            return "missing"
        with open(path, "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, or None if the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    k = t.get("kernels", {}).get(kernel)
    if not k or k.get("workload") != workload or k.get("source_digest") != kernel_source_digest(kernel):
        return None
    return k.get("dram_bytes_per_launch")

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
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


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(p, dtype: str, target_s: float = 10.0, step: str = "train") -> dict:
    """The oracle as it stands, on the host cores: the step on the full image
    (one image of the batch), repeated until about target_s of CPU time (at most
    5 repetitions)."""
    import oracle
    from dynamic_dilated_depthwise_gb300.inputs import Problem, SEEDS, make_inputs
    one = Problem(1, p.C, p.H, p.W, p.K, p.dilations)
    h = make_inputs(one, SEEDS.get(p.name, 1000), dtype, grad=step in ("train", "filter_train"),
                    taps=step in ("filter", "filter_train"))
    h = {k: v.double().numpy() for k, v in h.items()}
    bf = dtype == "bfloat16"
    oracle.build()
    reps, t_total = 0, 0.0
    while reps < 5 and (reps == 0 or t_total < target_s):
        t0 = time.perf_counter()
        if step in ("filter", "filter_train"):
            oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations)
            if step == "filter_train":
                oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
        else:
            oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)
        if step == "train":
            oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)
        t_total += time.perf_counter() - t0
        reps += 1
    px = reps * one.pixels
    what = {"train": "fwd+bwd", "forward": "forward", "filter": "filter-only",
            "filter_train": "filter-only fwd+bwd"}[step]
    return {"value": px / t_total / 1e6, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} x {what} of one {p.H}x{p.W} image (C={p.C}, K={p.K}, {dtype}-valued inputs, FP64 math)",
            "seconds": round(t_total, 3)}


def run_ours(args, world, rank, local):
    import torch
    from dynamic_dilated_depthwise_gb300 import binding, build
    from dynamic_dilated_depthwise_gb300.inputs import SEEDS, WORKLOADS, make_inputs

    build.build()
    lib = binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    p = WORKLOADS[args.workload]
    seed = SEEDS[p.name] + rank
    if args.batch is not None and args.batch != p.B:
        p = dataclasses.replace(p, B=args.batch, name=f"{p.name}_batch{args.batch}")
    dtype = args.dtype
    es = 2 if dtype == "bfloat16" else 4
    step_kind = args.step
    h = make_inputs(p, seed, dtype, grad=step_kind in ("train", "filter_train"),
                    taps=step_kind in ("filter", "filter_train"))
    if step_kind == "filter":
        h = {k: h[k] for k in ("x", "taps")}
    elif step_kind == "filter_train":
        h = {k: h[k] for k in ("x", "taps", "grad_out")}
    elif step_kind == "forward":
        h = {k: h[k] for k in ("x", "y", "weight", "bias")}
    d = {k: v.to(dev) for k, v in h.items()}
    flags = binding.DDPM_FLAG_CUDA_CORES if args.cuda_cores else binding.DDPM_FLAG_TF32_BACKWARD
    if args.tf32x3 and not args.cuda_cores:
        flags |= binding.DDPM_FLAG_TF32X3_FORWARD
    prob = binding.make_problem(p.B, p.C, p.H, p.W, p.K, p.dilations,
                                binding.DDPM_BFLOAT16 if dtype == "bfloat16" else binding.DDPM_FLOAT32, flags)
    out = torch.empty((p.B, 4 * p.C, p.H, p.W), dtype=d["x"].dtype, device=dev)
    dx, dy = torch.empty_like(d["x"]), torch.empty_like(d["x"])
    dw = torch.empty((p.O, p.C), dtype=d["x"].dtype, device=dev)
    db = torch.empty((p.O,), dtype=d["x"].dtype, device=dev)
    dtaps = torch.empty_like(d["taps"]) if step_kind == "filter_train" else None
    ws_bytes = binding.ddpm_backward_workspace_size(prob) if step_kind == "train" else 0
    if args.min_workspace and ws_bytes:
        ws_bytes = binding.ddpm_backward_workspace_min(prob)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    ptr = {k: v.data_ptr() for k, v in d.items()}
    import ctypes
    pref = ctypes.byref(prob)

    def step():
        if step_kind in ("filter", "filter_train"):
            s1, s2 = lib.ddpm_filter_pregenerated(pref, ptr["x"], ptr["taps"], out.data_ptr(), sh), 0
            if step_kind == "filter_train":
                s2 = lib.ddpm_filter_pregenerated_backward(pref, ptr["grad_out"], ptr["x"], ptr["taps"],
                                                           dx.data_ptr(), dtaps.data_ptr(), sh)
        else:
            s1 = lib.ddpm_forward(pref, ptr["x"], ptr["y"], ptr["weight"], ptr["bias"], out.data_ptr(), sh)
            s2 = 0
        if step_kind == "train":
            s2 = lib.ddpm_backward(pref, ptr["grad_out"], ptr["x"], ptr["y"], ptr["weight"], ptr["bias"],
                                   dx.data_ptr(), dy.data_ptr(), dw.data_ptr(), db.data_ptr(), ws.data_ptr(),
                                   ws.numel(), sh)
        if s1 or s2:
            raise RuntimeError(f"library error {binding.status_string(s1 or s2)}")

    if args.once:
        # profiling aid: W untimed steps, then one more step, and nothing else
        for _ in range(args.warmup + 1):
            step()
        torch.cuda.synchronize()
        assert binding.ddpm_get_device_error() == 0
        print(json.dumps({"once": step_kind, "workload": p.name, "dtype": dtype, "steps": args.warmup + 1}),
              flush=True)
        return None

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert binding.ddpm_get_device_error() == 0

    # ---- timed loop (value) ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(world, sum(step_ms))
    ms_per_step = total_ms / args.steps
    value = world * p.pixels / (ms_per_step * 1e-3) / 1e6

    # ---- steady state: the same steps back to back, no flush (inputs stay in L2) ----
    barrier(world)
    torch.cuda.synchronize()
    t_s0, t_s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_s0.record(stream)
    for _ in range(args.steps):
        step()
    t_s1.record(stream)
    torch.cuda.synchronize()
    steady_ms = max_over_ranks(world, t_s0.elapsed_time(t_s1)) / args.steps
    steady = {"value": round(world * p.pixels / (steady_ms * 1e-3) / 1e6, 3), "unit": UNIT,
              "ms_per_step": round(steady_ms, 5),
              "l2": "not flushed: steps back to back, inputs resident in L2 after the first"}

    # ---- traced loop: per-kernel device time on the launching stream ----
    binding.ddpm_trace_read()
    binding.ddpm_trace_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    binding.ddpm_trace_enable(False)
    recs = binding.ddpm_trace_read()
    per_kernel = {}
    for name, ms in recs:
        per_kernel.setdefault(name, []).append(ms)
    launches_per_step = len(recs) / args.steps
    peaks = load_peaks()
    splits = ws_bytes // (4 * p.O * (p.C + 1)) if ws_bytes else 1
    dominant = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    avg_ms = sum(per_kernel[dominant]) / len(per_kernel[dominant])
    bound, amount, kind = kernel_work(dominant, p, es, splits)
    if bound == "hbm":
        achieved, peak, unit = amount / (avg_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        achieved, peak, unit = amount / (avg_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    elif bound == "tensor_tf32":
        achieved, peak, unit = amount / (avg_ms * 1e-3) / 1e12, peaks["bf16_tflops"] * NOMINAL_TF32_OVER_BF16, "TFLOP/s"
    else:
        achieved, peak, unit = amount / (avg_ms * 1e-3) / 1e12, fp32_alu_tflops(peaks), "TFLOP/s"
    roof = {"bound": "tensor" if bound == "tensor_tf32" else bound, "kernel": dominant,
            "achieved": round(achieved, 3), "peak": round(peak, 1),
            "unit": unit, "frac": round(achieved / peak, 4),
            "traffic": stored_traffic(dominant, p.name),
            "peak_source": {"alu": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock",
                            "tensor_tf32": peaks["source"] + " bf16 x nominal tf32/bf16 (1.1/2.25)"}.get(
                                bound, peaks["source"]),
            "avg_launch_us": round(avg_ms * 1e3, 3),
            "work_per_launch": amount, "work_unit": kind}
    kernels = {k: {"launches_per_step": len(v) / args.steps, "avg_us": round(sum(v) / len(v) * 1e3, 3),
                   "share": round(sum(v) / sum(sum(x) for x in per_kernel.values()), 4)}
               for k, v in per_kernel.items()}
    sr = step_roofline_us(p, es, peaks, step_kind)
    step_roof = {"roofline_us": round(sr["roofline_us"], 3), "tensor_us": round(sr["tensor_us"], 3),
                 "hbm_us": round(sr["hbm_us"], 3), "measured_us": round(ms_per_step * 1e3, 3),
                 "frac": round(sr["roofline_us"] / (ms_per_step * 1e3), 4)}

    # ---- end to end through the C ABI: pinned host inputs in, results out ----
    # Every step copies all of its inputs in from pinned host memory and all of its
    # outputs back, inside the timed region.  The steps are pipelined two deep the way a
    # stream of batches would be: copy-in, compute and copy-out run on three streams over
    # double-buffered device tensors, so step i+1's inputs travel while step i computes
    # and step i-1's results return.
    e2e_steps = min(args.steps, 20)
    hin = {k: v.pin_memory() for k, v in h.items()}
    out_like = {"out": out, "dx": dx, "dy": dy, "dw": dw, "db": db}
    if step_kind == "filter_train":
        out_like = {"out": out, "dx": dx, "dtaps": dtaps}
    elif step_kind != "train":
        out_like = {"out": out}
    hout = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out_like.items()} for _ in range(2)]
    din = [d] + [{k: torch.empty_like(v) for k, v in d.items()}]
    dout = [out_like] + [{k: torch.empty_like(v) for k, v in out_like.items()}]
    bi = sum(v.numel() * v.element_size() for v in hin.values())
    bo = sum(v.numel() * v.element_size() for v in hout[0].values())
    s_in, s_c, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in_ready", "in_free", "c_done", "out_free")}

    def step_on(stream_c, pi, po):
        sc = stream_c.cuda_stream
        pp = {k: v.data_ptr() for k, v in pi.items()}
        if step_kind in ("filter", "filter_train"):
            s1, s2 = lib.ddpm_filter_pregenerated(pref, pp["x"], pp["taps"], po["out"].data_ptr(), sc), 0
            if step_kind == "filter_train":
                s2 = lib.ddpm_filter_pregenerated_backward(pref, pp["grad_out"], pp["x"], pp["taps"],
                                                           po["dx"].data_ptr(), po["dtaps"].data_ptr(), sc)
        else:
            s1 = lib.ddpm_forward(pref, pp["x"], pp["y"], pp["weight"], pp["bias"], po["out"].data_ptr(), sc)
            s2 = 0
        if step_kind == "train":
            s2 = lib.ddpm_backward(pref, pp["grad_out"], pp["x"], pp["y"], pp["weight"], pp["bias"],
                                   po["dx"].data_ptr(), po["dy"].data_ptr(), po["dw"].data_ptr(),
                                   po["db"].data_ptr(), ws.data_ptr(), ws.numel(), sc)
        if s1 or s2:
            raise RuntimeError(f"library error {binding.status_string(s1 or s2)}")

    def pipelined(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev["in_free"][b])
            with torch.cuda.stream(s_in):
                for k in hin:
                    din[b][k].copy_(hin[k], non_blocking=True)
            ev["in_ready"][b].record(s_in)
            s_c.wait_event(ev["in_ready"][b])
            if i >= 2:
                s_c.wait_event(ev["out_free"][b])
            step_on(s_c, din[b], dout[b])
            ev["in_free"][b].record(s_c)
            ev["c_done"][b].record(s_c)
            s_out.wait_event(ev["c_done"][b])
            with torch.cuda.stream(s_out):
                for k in hout[b]:
                    hout[b][k].copy_(dout[b][k], non_blocking=True)
            ev["out_free"][b].record(s_out)

    pipelined(2)                      # warm-up
    torch.cuda.synchronize()
    barrier(world)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(s_in)
    pipelined(e2e_steps)
    t_end.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, t_start.elapsed_time(t_end)) / e2e_steps
    e2e = {"value": round(world * p.pixels / (e2e_ms * 1e-3) / 1e6, 3), "unit": UNIT,
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 4),
           "pipeline": "2 steps deep: copy-in, compute and copy-out streams, double-buffered device tensors; "
                       "all inputs in and all outputs out every step"}
    assert binding.ddpm_get_device_error() == 0

    line = {"metric": STEP_METRIC[step_kind], "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if dtype == "bfloat16" else "f32",
            "data": "synthetic (seeded N(0,1) x, y, grad; weight N(0,1/C); bias N(0,0.01))",
            "config": {"workload": p.name, "B": p.B, "C": p.C, "H": p.H, "W": p.W, "K": p.K,
                       "dilations": list(p.dilations), "dtype": dtype,
                       "step": {"train": "ddpm_forward + ddpm_backward (dx, dy, dweight, dbias)",
                                "forward": "ddpm_forward (fused generator + filter)",
                                "filter": "ddpm_filter_pregenerated (taps given)",
                                "filter_train": "ddpm_filter_pregenerated + ddpm_filter_pregenerated_backward "
                                                "(dx, dtaps; taps given)"}[step_kind],
                       "l2": "flushed: 256 MiB write before each step, outside the timed events",
                       "flags": ("DDPM_FLAG_CUDA_CORES" if args.cuda_cores else
                                 "DDPM_FLAG_TF32_BACKWARD" + (" (FP32: dW/dbias partials on TF32 tensor cores; dX, dY "
                                                              "and the forward in IEEE FP32)" if dtype == "float32"
                                                              else " (ignored for bf16)")
                                 + (" | DDPM_FLAG_TF32X3_FORWARD (FP32 generator GEMM as three TF32 products, "
                                    "filter IEEE FP32)" if args.tf32x3 else "")),
                       "workspace_bytes": ws_bytes,
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "step_roofline": step_roof, "kernels": kernels,
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "e2e": e2e, "steady_state": steady, "wall_s_timed_loop": round(t_wall, 4)}
    line["clocks"] = clk.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, dtype, step=step_kind)
    return line


def run_reference(args, world, rank):
    """The CPU FP64 oracle on the host cores, timed as the reference arm."""
    if rank != 0:
        return None
    import oracle
    from dynamic_dilated_depthwise_gb300.inputs import Problem, SEEDS, WORKLOADS, make_inputs
    p = WORKLOADS[args.workload]
    kind = args.step
    rows = 16
    sample = Problem(1, p.C, rows, p.W, p.K, p.dilations)
    h = make_inputs(sample, SEEDS[p.name], args.dtype, grad=kind in ("train", "filter_train"),
                    taps=kind in ("filter", "filter_train"))
    h = {k: v.double().numpy() for k, v in h.items()}
    bf = args.dtype == "bfloat16"
    oracle.build()

    def step():
        # the same work as our arm's step, on the band
        if kind in ("filter", "filter_train"):
            oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations)
            if kind == "filter_train":
                oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
            return
        oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)
        if kind == "train":
            oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    ms = t / args.steps * 1e3
    value = sample.pixels / (ms * 1e-3) / 1e6
    what = {"train": "fwd+bwd", "forward": "forward", "filter": "filter-only",
            "filter_train": "filter-only fwd+bwd"}[kind]
    desc = f"{what} of a {rows}x{p.W} band (B=1, C={p.C}, K={p.K}) per step, FP64, {args.dtype}-valued inputs"
    return {"metric": STEP_METRIC[kind], "value": round(value, 4), "unit": UNIT, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": p.name, "B": p.B, "C": p.C, "H": p.H, "W": p.W, "K": p.K,
                       "dilations": list(p.dilations), "dtype": args.dtype, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def measure_fp32_peaks() -> dict:
    """FP32 FFMA throughput (the library's FMA-chain kernel on every SM) and cuBLAS TF32
    throughput (torch.matmul of two 8192 x 8192 FP32 matrices with TF32 allowed), each
    the best of a few timed runs: the denominators the CUDA-core and a TF32 path would
    be measured against."""
    import torch
    from dynamic_dilated_depthwise_gb300 import binding
    ffma = binding.ddpm_measure_ffma_tflops()
    n = 8192
    torch.backends.cuda.matmul.allow_tf32 = True
    a = torch.randn(n, n, device="cuda")
    b = torch.randn(n, n, device="cuda")
    for _ in range(3):
        torch.matmul(a, b)
    best = 1e30
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    tf32 = 2.0 * n ** 3 / (best * 1e-3) / 1e12
    return {"fp32_ffma_tflops": round(ffma, 2), "tf32_tflops": round(tf32, 1),
            "method": "FFMA: 8 independent fmaf chains per thread, 8 blocks of 256 per SM, best of 3; "
                      "TF32: torch.matmul 8192^3 FP32 with allow_tf32, best of 10"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--dtype", choices=("bfloat16", "float32"), default="bfloat16")
    ap.add_argument("--step", choices=("train", "forward", "filter", "filter_train"), default="train",
                    help="what one timed step runs (default: the fwd+bwd training step)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (faster runs)")
    ap.add_argument("--batch", type=int, default=None,
                    help="run the workload with this batch size instead of its own (larger inputs for profiling)")
    ap.add_argument("--min-workspace", action="store_true",
                    help="give the backward only the smallest workspace it accepts (the dW/dbias partials)")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="run the CUDA-core kernels (DDPM_FLAG_CUDA_CORES) instead of the tensor-core ones")
    ap.add_argument("--tf32x3", action="store_true",
                    help="FP32: compute the forward's generator GEMM as three TF32 tensor-core products "
                         "(DDPM_FLAG_TF32X3_FORWARD); the filter stays IEEE FP32")
    ap.add_argument("--once", action="store_true",
                    help="profiling aid: run --warmup untimed steps and one more step, print nothing else "
                         "(any --warmup >= 0); for one-kernel ncu captures")
    ap.add_argument("--peaks", action="store_true",
                    help="measure the FP32 FFMA and TF32 tensor peaks of this GPU and print them (one JSON line)")
    args = ap.parse_args()
    if args.warmup < 3 and not args.once:
        ap.error("--warmup must be at least 3")
    if args.batch is not None and args.batch < 1:
        ap.error("--batch must be at least 1")
    if args.peaks:
        print(json.dumps(measure_fp32_peaks()), flush=True)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
