#!/usr/bin/env python
"""NVFP4 linear-layer benchmark on one GB300 (or N independent replicas).

One step = the whole NVFP4 hot path of a 7B-shape MLP (hidden 4096, FFN 11008,
8192 tokens, no activation function) forward and backward, 12 kernel launches:

  dual(X: RN | RHT RN) . quantize_2d(W_up, +T) . GEMM  H  = X W_up^T
  dual(H: RN | RHT RN) . quantize_2d(W_down, +T) . GEMM  Y  = H W_down^T
  dual(dY: SR | RHT SR) . GEMM dH = dY W_down                (Dgrad down)
                          GEMM dW_down = dY^T H              (Wgrad down)
  dual(dH: SR | RHT SR) . GEMM dX = dH W_up                  (Dgrad up)
                          GEMM dW_up = dH^T X                (Wgrad up)

dual(.) is one read of a bf16 tensor that writes both its 1x16 row form (for
the Fprop/Dgrad GEMMs) and its Hadamard-transformed, transposed form (for the
Wgrad GEMMs), each bit-identical to the single-form quantizers.

Six GEMMs of 2*8192*11008*4096 flops.  `value` is NVFP4 TFLOP/s of the whole
step (all quantizers included) with inputs resident in HBM; `e2e` is the same
metric with the inputs copied from pinned host memory and the step's outputs
(Y, dX, dW_up, dW_down) copied back inside the timed region.  The inputs of a
step (~0.8 GB touched) exceed the 129 MB L2, so no flush is needed.

--impl reference times the CPU oracle (the plain C restatement) on a bounded
sample of the same workload and reports the same metric, extrapolated.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nvfp4_bit_quantized_quantize_gb300.step import MlpStep  # noqa: E402  (torch-free at import)

WORKLOAD = "mlp7b_fwd_bwd_h4096_f11008_t8192"
TOKENS, HIDDEN, FFN = 8192, 4096, 11008
GEMM_FLOPS = 2.0 * TOKENS * HIDDEN * FFN
N_GEMMS = 6
METRIC = "NVFP4 GEMM TFLOPS & quantize GB/s at 1 GB300, as fraction of roofline"
L2_BYTES = 129e6
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio (fp4 13.5 PF, bf16 2.25 PF)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def quant_bytes(kind: str, rows: int, cols: int) -> float:
    """Algorithmic HBM bytes of one quantizer launch: bf16 read once (twice when
    the tensor exceeds half the L2, since the tensor amax must be known before
    any code is written -- unless the amaxes are given), plus packed codes and
    scale bytes written."""
    n = rows * cols
    reads = 1 if kind.endswith("_from_amax") or 2 * n <= 0.5 * L2_BYTES else 2
    out = n / 2 + n / 16
    if kind in ("quantize_2d_t", "quantize_dual", "quantize_dual_from_amax"):
        out *= 2
    return reads * 2.0 * n + out


def source_hash(files):
    """Hash of the code of the given sources: comments and blank lines are
    left out, so that the committed counters stay tied to the kernel's code,
    not to its commentary."""
    h = hashlib.sha256()
    for f in files:
        for line in open(os.path.join(ROOT, f), encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


GEMM_SOURCES = ["nvfp4_bit_quantized_quantize_gb300/csrc/gemm.cu", "nvfp4_bit_quantized_quantize_gb300/csrc/gemm_common.cuh",
                "nvfp4_bit_quantized_quantize_gb300/csrc/device.cuh"]


def traffic_for(kernel: str, src_hash: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        t = json.load(open(path))[kernel]
        if t.get("source_hash") == src_hash:
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"nvfp4_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower().startswith("active")})
        sm = [r[0] for r in rows]
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------- our arm ----

class BenchStep(MlpStep):
    """The package's MlpStep at the 7B-MLP shape with two slots of inputs and
    results, plus pinned host copies of both for the end-to-end leg."""

    def __init__(self, dev):
        import numpy as np
        import torch

        import nvfp4_bit_quantized_quantize_gb300 as nv
        from nvfp4_bit_quantized_quantize_gb300 import synth

        seed = synth.WORKLOADS[WORKLOAD]["seed"]
        super().__init__(TOKENS, HIDDEN, FFN, seed, dev, slots=2)
        self.nv, self.dev = nv, dev
        host = synth.make_workload(WORKLOAD)
        bf = torch.bfloat16
        self.h_in = {k: torch.from_numpy(host[k].view(np.int16)).view(bf).pin_memory() for k in self.IN}
        for slot in self.inputs:
            for k, v in self.h_in.items():
                slot[k].copy_(v)
        self.h_out = [{k: torch.empty(v.shape, dtype=bf).pin_memory() for k, v in slot.items()}
                      for slot in self.outputs]
        torch.cuda.synchronize(dev)

    def h2d(self, slot):
        for k, v in self.h_in.items():
            self.inputs[slot][k].copy_(v, non_blocking=True)
        return sum(v.numel() * 2 for v in self.h_in.values())

    def d2h(self, slot):
        for k, v in self.outputs[slot].items():
            self.h_out[slot][k].copy_(v, non_blocking=True)
        return sum(v.numel() * 2 for v in self.outputs[slot].values())


def run_e2e(step, args, stream):
    """K steps through the public API with host buffers: every step copies its
    inputs from pinned host memory and its results back.  Copies run on their
    own streams into/out of two device slots, so step k's compute overlaps the
    input copy of step k+1 and the result copy of step k-1.  `args.warmup`
    untimed steps of the same pipeline run first (the first copies through
    fresh streams and buffers are slow)."""
    import torch

    if getattr(args, "warmup", 0) > 0:
        import types
        _e2e_steps(step, types.SimpleNamespace(steps=args.warmup), stream)
        torch.cuda.synchronize(step.dev)
    return _e2e_steps(step, args, stream)


def _e2e_steps(step, args, stream):
    import torch

    dev = step.dev
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready = [ev(), ev()]       # inputs of a slot landed
    in_free = [ev(), ev()]        # compute finished reading a slot's inputs
    out_ready = [ev(), ev()]      # compute finished writing a slot's results
    out_free = [ev(), ev()]       # results of a slot copied to the host
    side = step.side_stream()
    for e_ in in_free + out_free:
        e_.record(stream)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    h2d_s.wait_event(t0)
    h2d = d2h = 0
    for k in range(args.steps):
        sl = k % 2
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(in_free[sl])
            h2d = step.h2d(sl)
            in_ready[sl].record(h2d_s)
        stream.wait_event(in_ready[sl])
        stream.wait_event(out_free[sl])
        step.run_overlapped(sl, stream, side)   # joins its second stream before returning
        in_free[sl].record(stream)
        out_ready[sl].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[sl])
            d2h = step.d2h(sl)
            out_free[sl].record(d2h_s)
    stream.wait_stream(d2h_s)
    t1.record(stream)
    return t0, t1, h2d, d2h


def link_rates(step, stream, reps=5):
    """The host link alone, in the same run: one step's input copies (pinned
    host -> device) and result copies (device -> pinned host), each direction
    timed by itself and both at once on two streams (median of `reps`).  The
    pipelined end-to-end step cannot beat max(both directions at once, device
    step)."""
    import torch

    dev = step.dev
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(work):
        ts = []
        for _ in range(reps + 1):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for fn, st in work:
                st.wait_event(a)
                with torch.cuda.stream(st):
                    fn()
                e = torch.cuda.Event()
                e.record(st)
                stream.wait_event(e)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        return statistics.median(ts[1:])

    h_bytes = sum(v.numel() * 2 for v in step.h_in.values())
    d_bytes = sum(v.numel() * 2 for v in step.outputs[0].values())
    h_ms = timed([(lambda: step.h2d(0), s1)])
    d_ms = timed([(lambda: step.d2h(0), s2)])
    both_ms = timed([(lambda: step.h2d(0), s1), (lambda: step.d2h(0), s2)])
    return {"h2d_ms": round(h_ms, 4), "h2d_gbs": round(h_bytes / (h_ms * 1e-3) / 1e9, 1),
            "d2h_ms": round(d_ms, 4), "d2h_gbs": round(d_bytes / (d_ms * 1e-3) / 1e9, 1),
            "both_ms": round(both_ms, 4),
            "how": "one step's pinned copies (cudaMemcpyAsync per buffer), each direction alone and both at once "
                   "on two streams, median of 5"}


def bind_host_to_gpu_node(dev_index: int):
    """Run this process on the CPUs attached to the GPU (the PCI device's
    local_cpulist in sysfs), so that the pinned host buffers, which land on
    the allocating thread's memory node, sit next to the GPU's own host link
    instead of behind a CPU-to-CPU hop.  Returns the CPU list, or None when
    sysfs does not give one."""
    import torch

    p = torch.cuda.get_device_properties(dev_index)
    path = f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0/local_cpulist"
    try:
        txt = open(path).read().strip()
    except OSError:
        return None
    cpus = set()
    for part in txt.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part:
            cpus.add(int(part))
    cpus &= os.sched_getaffinity(0)
    if not cpus:
        return None
    os.sched_setaffinity(0, cpus)
    return txt


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: with N replicas the job ends when the last one
    does.  One all-reduce MAX of a single float64 (on `device`: the rank's GPU
    under NCCL, the CPU under gloo)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step_per_rank: float, ms_per_step: float) -> float:
    """Whole-job throughput of N weak-scaled replicas: every rank does one
    step's flops in the slowest rank's step time."""
    return world * flops_per_step_per_rank / (ms_per_step * 1e-3) / 1e12


def check_status(step, when: str) -> None:
    """Both workspaces' device status (the step's second stream has its own)."""
    for ws in (step.ws, step.ws_side):
        st = step.nv.nvfp4_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status after {when}: {step.nv.nvfp4_status_str(st)}")


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from __graft_entry__ import build
    build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    host_cpus = bind_host_to_gpu_node(local_rank)
    step = BenchStep(dev)
    launches = step.launches()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    side = step.side_stream()
    for _ in range(args.warmup):
        step.run_overlapped(0, stream, side)
    for _ in range(args.warmup):
        for l in launches:
            l.fn()
    check_status(step, "warm-up")
    barrier()

    # ---- timed region: inputs resident in HBM; the step's schedule (the
    # weight-gradient GEMMs on a second stream), no events between launches ----
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t0.record(stream)
    for k in range(args.steps):
        step.run_overlapped(0, stream, side)
    t1.record(stream)
    barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    check_status(step, "timed steps")

    # ---- per-kernel durations: the same K steps again, the twelve launches
    # in order on one stream with one event pair around each ----
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in launches]
           for _ in range(args.steps)]
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    barrier()
    s0.record(stream)
    for k in range(args.steps):
        for l, (a, b) in zip(launches, evs[k]):
            a.record(stream)
            l.fn()
            b.record(stream)
    s1.record(stream)
    barrier()
    clk = clocks.stop()
    ms_seq = max_over_ranks(s0.elapsed_time(s1), world, dev) / args.steps
    check_status(step, "per-kernel steps")

    per_kind = {}
    for k in range(args.steps):
        for l, (a, b) in zip(launches, evs[k]):
            per_kind.setdefault((l.kind, l.shape), []).append(a.elapsed_time(b))
    ms_step = ms_total / args.steps
    flops_step = N_GEMMS * GEMM_FLOPS
    value = job_tflops(world, flops_step, ms_step)

    pk = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    gemm_ms = [t for (kind, _), ts in per_kind.items() if kind == "gemm" for t in ts]
    gemm_avg = statistics.mean(gemm_ms)
    gemm_tflops = GEMM_FLOPS / (gemm_avg * 1e-3) / 1e12
    kernels = {}
    for (kind, shape), ts in per_kind.items():
        avg = statistics.mean(ts)
        key = f"{kind}[{'x'.join(str(s) for s in shape)}]"
        if kind == "gemm":
            f = 2.0 * shape[0] * shape[1] * shape[2]
            kernels[key] = {"ms": round(avg, 4), "TFLOP/s": round(f / (avg * 1e-3) / 1e12, 1),
                            "frac": round(f / (avg * 1e-3) / 1e12 / fp4_peak, 3)}
        else:
            byts = quant_bytes(kind, shape[1], shape[2])
            gbs = byts / (avg * 1e-3) / 1e9
            kernels[key] = {"ms": round(avg, 4), "GB/s": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 3)}
    q_ms = sum(statistics.mean(ts) for (kind, _), ts in per_kind.items() if kind != "gemm")
    q_bytes = sum(quant_bytes(kind, sh[1], sh[2]) * len(ts) / args.steps
                  for (kind, sh), ts in per_kind.items() if kind != "gemm")
    step_kernel_ms = sum(statistics.mean(ts) * len(ts) / args.steps for ts in per_kind.values())

    src_hash = source_hash(GEMM_SOURCES)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 codes, e4m3 block scales, f32 tensor scale) -> f32 accumulate -> bf16",
        "data": "synthetic (seeded N(0,1)/N(0,0.02)/N(0,1e-3), 0.1% outliers x100 on X)",
        "config": {"workload": WORKLOAD, "tokens": TOKENS, "hidden": HIDDEN, "ffn": FFN,
                   "gemms_per_step": N_GEMMS, "launches_per_step": len(launches),
                   "l2": "inputs larger than L2 (about 0.8 GB touched per step), no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "nvf4_gemm_pair_kernel", "achieved": round(gemm_tflops, 1),
                     "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(gemm_tflops / fp4_peak, 4),
                     "traffic": traffic_for("nvf4_gemm_pair_kernel", src_hash),
                     "peak_note": f"{pk['source']} bf16 burst {pk['bf16_tflops']} x {FP4_OVER_BF16} (fp4/bf16 nominal)",
                     "algorithmic_flops_per_launch": GEMM_FLOPS},
        "quantize": {"GB/s": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
                     "frac": round(q_bytes / (q_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
                     "peak_gbs": pk["hbm_gbs"], "ms_per_step": round(q_ms, 4)},
        "kernels": kernels,
        "kernel_ms_per_step": round(step_kernel_ms, 4),
        "schedule": {"timed": "weight-gradient GEMMs on a second stream beside the data-gradient work",
                     "kernels_from": "a second pass of the same steps, launches in order on one stream with an "
                                     "event pair around each (roofline and kernels come from it)",
                     "sequential_ms_per_step": round(ms_seq, 4)},
        "gpu_launches": len(launches) * args.steps,
        "clocks": clk,
    }

    # ---- end to end: pinned host inputs in, results out, every step ----
    if not args.no_e2e:
        # first touches of the pinned host buffers are slow: both slots' copy
        # paths are exercised (and the link timed) before the timed e2e steps
        link = link_rates(step, stream)
        for slot in (0, 1):
            step.h2d(slot)
            step.d2h(slot)
        barrier()
        e0, e1, h2d, d2h = run_e2e(step, args, stream)
        barrier()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, dev)
        check_status(step, "end-to-end steps")
        link["bound_ms_per_step"] = round(max(link["both_ms"], ms_step), 4)
        line["e2e"] = {"value": round(job_tflops(world, flops_step, ms_e2e / args.steps), 2),
                       "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(ms_e2e / args.steps, 4),
                       "note": "pinned host inputs copied in and results copied out every step; copies on "
                               "separate streams overlap the neighbouring steps' compute (two device slots)",
                       "host_cpus": host_cpus, "link": link}

    if not args.no_extras:
        line["extras"] = measure_extras(step, stream, pk)
        line["configs"] = measure_configs(step, stream, pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    return line


def _event_ms(fn, stream, reps=10, warmup=3):
    """Mean CUDA-event time of fn() on `stream` after warm-up."""
    import torch

    for _ in range(warmup):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _flushed_ms(fn, stream, flush, reps=20, warmup=5):
    """Median CUDA-event time of fn() on `stream`, the L2 flushed (a buffer of
    twice its size written) before every launch; the flush is outside the
    events."""
    import torch

    evs = []
    for i in range(warmup + reps):
        flush.fill_(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if i >= warmup:
            evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def measure_configs(step, stream, pk):
    """The other workloads' kernels alone (5 warm-up launches, median of 20,
    L2 flushed before each launch): the quantize sweep (1024^2, 4096^2,
    8192^2, RN and SR), the 2-D weight Fprop (W 20480x5120 2-D with
    transpose, X 8192x5120 RN, GEMM 8192x20480x5120) and the RHT+SR Wgrad
    (dY and X 16384x5120, GEMM 5120x5120x16384).  Inputs are N(0,1)
    (N(0,0.02) for W, N(0,1e-3) for dY) drawn on the device."""
    import torch

    nv = step.nv
    dev = step.dev
    ws = step.ws
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.int32, device=dev)
    out = {}

    def qline(kind, rows, cols, ms):
        gbs = quant_bytes(kind, rows, cols) / (ms * 1e-3) / 1e9
        return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 3)}

    def gline(M, N, K, ms):
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac": round(tf / fp4_peak, 3)}

    # tiny linear layer (X, W 256x256, N(0,1) with 0.5% x50, seed 0): two RN
    # quantizations and the 256^3 GEMM; latency-bound, reported, not graded
    import numpy as np

    from nvfp4_bit_quantized_quantize_gb300 import synth
    wl = synth.make_workload("tiny_linear_256")
    n1 = 256
    X1, W1 = (torch.from_numpy(wl[k].view(np.int16)).to(dev).view(torch.bfloat16) for k in ("X", "W"))
    xq1, wq1 = nv.alloc_quantized(n1, n1, dev), nv.alloc_quantized(n1, n1, dev)
    d1 = torch.empty((n1, n1), dtype=torch.bfloat16, device=dev)
    qx = lambda: nv.nvfp4_quantize(X1, n1, n1, n1, nv.RN, 0, *xq1, ws)
    qw = lambda: nv.nvfp4_quantize(W1, n1, n1, n1, nv.RN, 0, *wq1, ws)
    g1 = lambda: nv.nvfp4_gemm(*xq1, *wq1, n1, n1, n1, d1, n1, nv.OUT_BF16, ws)
    out["tiny_linear_256/quantize_1x16[rnx256x256]"] = qline("quantize_1x16", n1, n1, _flushed_ms(qx, stream, flush))
    out["tiny_linear_256/gemm[256x256x256]"] = gline(n1, n1, n1, _flushed_ms(g1, stream, flush))
    ms = _flushed_ms(lambda: (qx(), qw(), g1()), stream, flush)
    out["tiny_linear_256/layer[3 launches]"] = {"ms": round(ms, 4), "note": "quantize X, quantize W, GEMM; "
                                                "latency-bound (reported, not graded)"}
    del X1, W1, xq1, wq1, d1

    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    for n in (1024, 4096, 8192):
        x = torch.randn((n, n), generator=gen, device=dev).to(torch.bfloat16)
        q, sf, g = nv.alloc_quantized(n, n, dev)
        for mode, tag in ((nv.RN, "rn"), (nv.SR, "sr")):
            ms = _flushed_ms(lambda: nv.nvfp4_quantize(x, n, n, n, mode, 7, q, sf, g, ws), stream, flush)
            out[f"quantize_sweep/quantize_1x16[{tag}x{n}x{n}]"] = qline("quantize_1x16", n, n, ms)
        del x, q, sf, g
    # 2-D weight Fprop
    M, N, K = 8192, 20480, 5120
    w = (torch.randn((N, K), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    x = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
    wq, wqT, xq = nv.alloc_quantized(N, K, dev), nv.alloc_quantized(K, N, dev), nv.alloc_quantized(M, K, dev)
    ms = _flushed_ms(lambda: nv.nvfp4_quantize_2d(w, N, K, K, wq[0], wq[1], wqT[0], wqT[1], wq[2], ws), stream,
                     flush)
    out[f"fprop_w2d/quantize_2d_t[{N}x{K}]"] = qline("quantize_2d_t", N, K, ms)
    ms = _flushed_ms(lambda: nv.nvfp4_quantize(x, M, K, K, nv.RN, 0, *xq, ws), stream, flush)
    out[f"fprop_w2d/quantize_1x16[rnx{M}x{K}]"] = qline("quantize_1x16", M, K, ms)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ms = _flushed_ms(lambda: nv.nvfp4_gemm(xq[0], xq[1], xq[2], wq[0], wq[1], wq[2], M, N, K, d, N,
                                           nv.OUT_BF16, ws), stream, flush)
    out[f"fprop_w2d/gemm[{M}x{N}x{K}]"] = gline(M, N, K, ms)
    del w, x, wq, wqT, xq, d
    # RHT + SR Wgrad
    T, C = 16384, 5120
    dy = (torch.randn((T, C), generator=gen, device=dev) * 1e-3).to(torch.bfloat16)
    x = torch.randn((T, C), generator=gen, device=dev).to(torch.bfloat16)
    dyT, xT = nv.alloc_quantized(C, T, dev), nv.alloc_quantized(C, T, dev)
    ms = _flushed_ms(lambda: nv.nvfp4_rht_quantize(dy, T, C, C, 4, nv.SR, 3, *dyT, ws), stream, flush)
    out[f"wgrad_rht_sr/rht_quantize[srx{T}x{C}]"] = qline("rht_quantize", T, C, ms)
    ms = _flushed_ms(lambda: nv.nvfp4_rht_quantize(x, T, C, C, 4, nv.SR, 5, *xT, ws), stream, flush)
    out[f"wgrad_rht_sr/rht_quantize[srx{T}x{C}]/X"] = qline("rht_quantize", T, C, ms)
    d = torch.empty((C, C), dtype=torch.bfloat16, device=dev)
    ms = _flushed_ms(lambda: nv.nvfp4_gemm(dyT[0], dyT[1], dyT[2], xT[0], xT[1], xT[2], C, C, T, d, C,
                                           nv.OUT_BF16, ws), stream, flush)
    out[f"wgrad_rht_sr/gemm[{C}x{C}x{T}]"] = gline(C, C, T, ms)
    del dy, x, dyT, xT, d, flush
    st = nv.nvfp4_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after config kernels: {nv.nvfp4_status_str(st)}")
    return out


def cublaslt_nvfp4(a, b, M, N, K):
    """cuBLASLt's block-scaled NVFP4 GEMM through torch._scaled_mm on codes and
    128x4-atom scale bytes laid out as this library writes them (the layout
    the library call reads as its swizzled block scales).  Returns the call."""
    import torch

    rup = lambda x, m: (x + m - 1) // m * m
    A = a[0].view(torch.float4_e2m1fn_x2)
    B = b[0].view(torch.float4_e2m1fn_x2)
    SA = a[1].view(torch.float8_e4m3fn).view(rup(M, 128), rup(K // 16, 4))
    SB = b[1].view(torch.float8_e4m3fn).view(rup(N, 128), rup(K // 16, 4))
    return lambda: torch._scaled_mm(A, B.t(), SA, SB, out_dtype=torch.bfloat16)


def measure_extras(step, stream, pk):
    """Kernels beside the step, each timed alone (not part of `value`):
    the quantization-noise meter on H's forward form, a GEMM with ragged
    M, N, K, the MXFP4 quantizer and GEMM (the comparison format), and cuBLAS
    bf16 matmul on the step's six GEMM shapes for context."""
    import torch

    nv = step.nv
    T, D, F = TOKENS, HIDDEN, FFN
    dev = step.dev
    out = {}
    # noise meter: reads H (bf16) + its codes + scales once: 2.5625 B/element
    sums = torch.empty(2, dtype=torch.float64, device=dev)
    q, sf, g = step.hq
    ms = _event_ms(lambda: nv.nvfp4_quant_noise(step.H, T, F, F, q, sf, g, sums), stream)
    byts = 2.5625 * T * F
    out["quant_noise[8192x11008]"] = {"ms": round(ms, 4), "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                      "frac": round(byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
                                      "norm_ratio": round(float((sums[1] / sums[0]).sqrt()), 3)}
    # binary32 output (the strict-check form) on the up-projection Fprop operands
    d32 = torch.empty((T, F), dtype=torch.float32, device=dev)
    ms = _event_ms(lambda: nv.nvfp4_gemm(*step.xq, *step.wuq, T, F, D, d32, F, nv.OUT_F32, step.ws), stream)
    out["gemm_f32_out[8192x11008x4096]"] = {"ms": round(ms, 4),
                                             "TFLOP/s": round(GEMM_FLOPS / (ms * 1e-3) / 1e12, 1),
                                             "frac": round(GEMM_FLOPS / (ms * 1e-3) / 1e12
                                                           / (pk["bf16_tflops"] * FP4_OVER_BF16), 3)}
    del d32
    # ragged GEMM: every dimension off the tile grid
    M, N, K = 8000, 11000, 4064
    a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev)
    b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev)
    sfa = torch.randint(0x30, 0x48, (nv.nvfp4_sf_bytes(M, K),), dtype=torch.uint8, device=dev)
    sfb = torch.randint(0x30, 0x48, (nv.nvfp4_sf_bytes(N, K),), dtype=torch.uint8, device=dev)
    one = torch.ones(1, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ms = _event_ms(lambda: nv.nvfp4_gemm(a, sfa, one, b, sfb, one, M, N, K, d, N, nv.OUT_BF16, step.ws), stream)
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    out[f"gemm_ragged[{M}x{N}x{K}]"] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1)}
    del a, b, sfa, sfb, d
    # MXFP4 comparison format: one streaming quantizer pass over H, and the
    # up-projection Fprop GEMM on MXFP4 operands of X and W_up
    mq = torch.empty((T, F // 2), dtype=torch.uint8, device=dev)
    msf = torch.empty((nv.nvfp4_sf_bytes(T, F),), dtype=torch.uint8, device=dev)
    ms = _event_ms(lambda: nv.nvfp4_mxfp4_quantize(step.H, T, F, F, mq, msf, step.ws), stream)
    byts = (2.0 + 0.5 + 1.0 / 32) * T * F
    out["mxfp4_quantize[8192x11008]"] = {"ms": round(ms, 4), "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                         "frac": round(byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)}
    xa = (torch.empty((T, D // 2), dtype=torch.uint8, device=dev),
          torch.empty((nv.nvfp4_sf_bytes(T, D),), dtype=torch.uint8, device=dev))
    wb = (torch.empty((F, D // 2), dtype=torch.uint8, device=dev),
          torch.empty((nv.nvfp4_sf_bytes(F, D),), dtype=torch.uint8, device=dev))
    nv.nvfp4_mxfp4_quantize(step.inputs[0]["X"], T, D, D, xa[0], xa[1], step.ws)
    nv.nvfp4_mxfp4_quantize(step.inputs[0]["W_up"], F, D, D, wb[0], wb[1], step.ws)
    ms = _event_ms(lambda: nv.nvfp4_mxfp4_gemm(xa[0], xa[1], wb[0], wb[1], T, F, D, step.H, F, nv.OUT_BF16,
                                               step.ws), stream)
    out["mxfp4_gemm[8192x11008x4096]"] = {"ms": round(ms, 4),
                                           "TFLOP/s": round(GEMM_FLOPS / (ms * 1e-3) / 1e12, 1)}
    del mq, msf, xa, wb
    # cuBLASLt's NVFP4 GEMM on the up-projection Fprop shape (context: the
    # vendor library on the same operands' codes and block scales)
    key = "cublaslt_nvfp4[8192x11008x4096]"
    try:
        fn = cublaslt_nvfp4(step.xq[:2], step.wuq[:2], T, F, D)
        fn()
        ms = _event_ms(fn, stream, reps=5)
        out[key] = {"ms": round(ms, 4), "TFLOP/s": round(GEMM_FLOPS / (ms * 1e-3) / 1e12, 1),
                    "note": "torch._scaled_mm, bf16 out, block scales only (no tensor scale); context, not this "
                            "library"}
    except Exception as e:  # a torch without NVFP4 _scaled_mm
        out[key] = {"unavailable": str(e).splitlines()[0][:160]}
    # cuBLAS bf16 on the same six GEMMs (context: the unquantized layer)
    shapes = [(T, F, D), (T, D, F), (T, F, D), (D, F, T), (T, D, F), (F, D, T)]
    tot = 0.0
    for (m, n, k) in shapes:
        x = torch.randn((m, k), dtype=torch.bfloat16, device=dev)
        w = torch.randn((n, k), dtype=torch.bfloat16, device=dev)
        tot += _event_ms(lambda: torch.matmul(x, w.t()), stream, reps=5)
        del x, w
    out["cublas_bf16_six_gemms"] = {"ms": round(tot, 4),
                                    "TFLOP/s": round(N_GEMMS * GEMM_FLOPS / (tot * 1e-3) / 1e12, 1)}
    st = nv.nvfp4_device_status(step.ws)
    if st != 0:
        raise RuntimeError(f"device status after extras: {nv.nvfp4_status_str(st)}")
    return out


# ------------------------------------------------------- CPU oracle arm ----

def host_cores() -> int:
    """Host CPUs this process may run on (the affinity mask; nproc's count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_estimate(budget_s: float, threads: int = 1):
    """Time the oracle on bounded samples of every kind of launch of the step
    (each sample sized to about a fifth of budget_s) and extrapolate the time of
    one full step.  With threads > 1 every sample runs as `threads` row slices
    at once, one oracle call per host thread (the oracle's C code runs outside
    the interpreter lock), and the per-element time is the wall time over all
    slices.  Returns (seconds, sample description, samples timed)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle as O
    from nvfp4_bit_quantized_quantize_gb300 import synth

    T, D, F = TOKENS, HIDDEN, FFN
    share = budget_s / 5.0
    pool = cf.ThreadPoolExecutor(threads) if threads > 1 else None
    timed = [0]

    def per_unit(make, run, units, lo=1):
        """Grow the sample until one run (of `threads` slices) takes about
        `share` seconds."""
        n = lo
        while True:
            args_ = [make(n) for _ in range(threads)]
            t = time.perf_counter()
            if pool is None:
                run(args_[0])
            else:
                list(pool.map(run, args_))
            dt = time.perf_counter() - t
            timed[0] += 1
            if dt >= share * 0.5 or n >= (1 << 20):
                return dt / (units(n) * threads), n
            n = max(n * 2, int(n * share / max(dt, 1e-4) * 0.9))

    rng = np.random.default_rng(0)
    mk_x = lambda r: synth.normal_bf16((r, D), 4, 0, 1.0, 0.0, 0.001, 100.0)
    t_rn, r_rn = per_unit(mk_x, lambda x: O.quantize(x, O.RN), lambda r: r * D, 16)
    t_sr, r_sr = per_unit(mk_x, lambda x: O.quantize(x, O.SR, 1), lambda r: r * D, 16)
    t_2d, r_2d = per_unit(lambda r: synth.normal_bf16((16 * r, D), 4, 1, 0.02), O.quantize_2d,
                          lambda r: 16 * r * D, 1)
    t_rht, c_rht = per_unit(lambda c: synth.normal_bf16((T, 8 * c), 4, 2, 1e-3),
                            lambda x: O.rht_quantize(x, 5, O.SR, 1), lambda c: T * 8 * c, 1)
    K = D
    qa = rng.integers(0, 256, (64, K // 2), dtype=np.uint8)
    sa = np.full(O.sf_bytes(64, K), 0x38, np.uint8)
    t_mac, n_out = per_unit(lambda n: (np.arange(n) % 64, (np.arange(n) * 7) % 64),
                            lambda mn: O.gemm_f64_sampled(qa, sa, 1.0, qa, sa, 1.0, 64, 64, K, mn[0], mn[1]),
                            lambda n: n * K, 8)
    if pool is not None:
        pool.shutdown()

    el = lambda r, c: r * c
    quant = (t_rn * (el(T, D) + el(T, F)) + t_sr * (el(T, D) + el(T, F)) + t_2d * (el(F, D) + el(D, F))
             + t_rht * (el(T, D) * 2 + el(T, F) * 2))
    total = quant + t_mac * (N_GEMMS * GEMM_FLOPS / 2)
    per = f"{threads} x " if threads > 1 else ""
    sample = (f"oracle timed on {per}{r_rn}x{D} (1x16 RN), {per}{r_rn}x{D} (1x16 SR), {per}{16 * r_2d}x{D} "
              f"(2-D), {per}{T}x{8 * c_rht} (RHT+SR) slices and {per}{n_out} GEMM outputs at K={K}; "
              f"per-element and per-MAC times extrapolated to the full step ({N_GEMMS} GEMMs; the 1x16, "
              f"Hadamard and 2-D quantizations of the step's 4 dual and 2 weight launches)")
    return total, sample, timed[0]


def cpu_baseline(budget_s: float = 15.0):
    """The oracle on one host thread (the headline `value`, `cores` = 1) and
    on every host core (`all_cores`), each on bounded samples of the step."""
    t = time.perf_counter()
    est, sample, _ = oracle_step_estimate(budget_s)
    wall = time.perf_counter() - t
    ncores = host_cores()
    out = {"value": N_GEMMS * GEMM_FLOPS / est / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": sample + f" (measured in {wall:.1f} s, single thread)",
           "extrapolated": True, "extrapolated_step_s": round(est, 1), "host_nproc": ncores}
    if ncores > 1:
        t = time.perf_counter()
        est_n, sample_n, _ = oracle_step_estimate(budget_s, threads=ncores)
        wall = time.perf_counter() - t
        out["all_cores"] = {"value": N_GEMMS * GEMM_FLOPS / est_n / 1e12, "unit": "TFLOP/s", "cores": ncores,
                            "sample": sample_n + f" (measured in {wall:.1f} s, {ncores} threads)",
                            "extrapolated_step_s": round(est_n, 1)}
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on this host, one thread.  Each
    "step" is a bounded sample of the workload from which a full step's time
    is extrapolated; the line says so (`extrapolated`, `samples_timed`)."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    ests = []
    sample = ""
    n_timed = 0
    t0 = time.perf_counter()
    for i in range(args.warmup + args.steps):
        est, sample, k = oracle_step_estimate(budget_s=args.cpu_budget / 3)
        if i >= args.warmup:
            ests.append(est)
            n_timed += k
    wall = time.perf_counter() - t0
    s_step = statistics.median(ests)
    value = N_GEMMS * GEMM_FLOPS / s_step / 1e12
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 decisions, f64 GEMM accumulation (oracle)",
            "data": "synthetic", "config": {"workload": WORKLOAD, "tokens": TOKENS, "hidden": HIDDEN, "ffn": FFN},
            "extrapolated": True,
            "extrapolation": (f"each of the {args.steps} timed steps is {n_timed // max(args.steps, 1)} bounded "
                              f"oracle samples (about {args.cpu_budget / 3:.0f} s of CPU work) whose per-element "
                              f"and per-MAC times are scaled to one full step; ms_per_step is that estimate, "
                              f"not a measured step ({wall:.1f} s of wall time in all)"),
            "samples_timed": n_timed,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "host_nproc": host_cores()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------- one kernel, for ncu ----

def run_case(argv):
    """One library kernel on synthetic device data, for profiler captures:

      --case gemm M N K [f32]      random codes, E4M3 scales in [2^-6, 2^2)
      --case gemm_amax M N K       the same, bf16 output and its two maxima
      --case cublaslt M N K        cuBLASLt's NVFP4 GEMM on the same kind of data (context)
      --case quantize ROWS COLS rn|sr
      --case quantize_2d ROWS COLS
      --case rht T C rn|sr
      --case dual T C rn|sr
      --case dual_amax T C rn|sr   the dual quantizer with both amaxes given
      --case noise ROWS COLS

    Two warm-up launches, then --steps launches; prints the mean CUDA-event
    time per launch (not a benchmark while a profiler is attached)."""
    import torch

    import nvfp4_bit_quantized_quantize_gb300 as nv
    from __graft_entry__ import build

    build()
    kind, rest = argv[0], argv[1:]
    reps = CASE_REPS[0]
    torch.manual_seed(0)
    ws = nv.alloc_workspace()
    if kind == "cublaslt":
        M, N, K = (int(v) for v in rest[:3])
        a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda")
        b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda")
        sfa = torch.randint(0x18, 0x48, (nv.nvfp4_sf_bytes(M, K),), dtype=torch.uint8, device="cuda")
        sfb = torch.randint(0x18, 0x48, (nv.nvfp4_sf_bytes(N, K),), dtype=torch.uint8, device="cuda")
        fn = cublaslt_nvfp4((a, sfa), (b, sfb), M, N, K)
        what = f"cublaslt {M}x{N}x{K}"
        work = lambda ms: f"{2 * M * N * K / ms / 1e9:.1f} TFLOP/s"
    elif kind in ("gemm", "gemm_amax"):
        M, N, K = (int(v) for v in rest[:3])
        f32 = kind == "gemm" and len(rest) > 3 and rest[3] == "f32"
        a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda")
        b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda")
        sfa = torch.randint(0x18, 0x48, (nv.nvfp4_sf_bytes(M, K),), dtype=torch.uint8, device="cuda")
        sfb = torch.randint(0x18, 0x48, (nv.nvfp4_sf_bytes(N, K),), dtype=torch.uint8, device="cuda")
        one = torch.ones(1, device="cuda")
        d = torch.empty((M, N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        if kind == "gemm":
            fn = lambda: nv.nvfp4_gemm(a, sfa, one, b, sfb, one, M, N, K, d, N,
                                       nv.OUT_F32 if f32 else nv.OUT_BF16, ws)
        else:
            am = torch.zeros(2, dtype=torch.float32, device="cuda")
            fn = lambda: nv.nvfp4_gemm_amax(a, sfa, one, b, sfb, one, M, N, K, d, N, 5, am, ws)
        what = f"{kind} {M}x{N}x{K}{' f32' if f32 else ''}"
        work = lambda ms: f"{2 * M * N * K / ms / 1e9:.1f} TFLOP/s"
    else:
        R, C = int(rest[0]), int(rest[1])
        mode = nv.SR if (len(rest) > 2 and rest[2] == "sr") else nv.RN
        x = torch.randn((R, C), dtype=torch.bfloat16, device="cuda")
        if kind == "quantize":
            q, sf, g = nv.alloc_quantized(R, C)
            fn = lambda: nv.nvfp4_quantize(x, R, C, C, mode, 1, q, sf, g, ws)
        elif kind == "quantize_2d":
            q, sf, g = nv.alloc_quantized(R, C)
            qT, sfT, _ = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_quantize_2d(x, R, C, C, q, sf, qT, sfT, g, ws)
        elif kind == "rht":
            q, sf, g = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_rht_quantize(x, R, C, C, 5, mode, 1, q, sf, g, ws)
        elif kind == "dual":
            q, sf, g = nv.alloc_quantized(R, C)
            qT, sfT, gT = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_quantize_dual(x, R, C, C, mode, 1, q, sf, g, 5, mode, 2, qT, sfT, gT, ws)
        elif kind == "dual_amax":
            q, sf, g = nv.alloc_quantized(R, C)
            qT, sfT, gT = nv.alloc_quantized(C, R)
            am = torch.tensor([4.5, 4.0], dtype=torch.float32, device="cuda")  # about the maxima of N(0,1)
            fn = lambda: nv.nvfp4_quantize_dual_from_amax(x, R, C, C, am, mode, 1, q, sf, g, 5, mode, 2, qT, sfT,
                                                          gT, ws)
        elif kind == "noise":
            q, sf, g = nv.alloc_quantized(R, C)
            nv.nvfp4_quantize(x, R, C, C, nv.RN, 0, q, sf, g, ws)
            sums = torch.empty(2, dtype=torch.float64, device="cuda")
            fn = lambda: nv.nvfp4_quant_noise(x, R, C, C, q, sf, g, sums)
        else:
            raise SystemExit(run_case.__doc__)
        what = f"{kind} {R}x{C}{' sr' if mode == nv.SR else ''}"
        byts = 2.5625 * R * C if kind == "noise" else quant_bytes(
            {"quantize": "quantize_1x16", "quantize_2d": "quantize_2d_t", "rht": "rht_quantize",
             "dual": "quantize_dual", "dual_amax": "quantize_dual_from_amax"}[kind], R, C)
        work = lambda ms: f"{byts / ms / 1e6:.1f} GB/s algorithmic"
    stream = torch.cuda.current_stream()
    ms = _event_ms(fn, stream, reps=reps, warmup=2)
    st = nv.nvfp4_device_status(ws)
    if st != 0:
        raise SystemExit(f"device status {nv.nvfp4_status_str(st)}")
    print(f"{what}: {ms:.4f} ms per launch, {work(ms)}")


CASE_REPS = [3]


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--case", nargs="+", metavar="ARG",
                    help="run one kernel for a profiler capture instead of the benchmark "
                         "(gemm M N K [f32] | quantize R C rn|sr | quantize_2d R C | rht T C rn|sr | "
                         "dual T C rn|sr | noise R C); --steps launches after 2 warm-up launches")
    args = ap.parse_args()
    if args.case:
        CASE_REPS[0] = args.steps
        run_case(args.case)
        return
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
