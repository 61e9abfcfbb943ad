"""Benchmark of the tcgen05 GEMM library on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-variants]

Headline workload: bf16 GEMM M = N = K = 8192, A ~ N(0,1), B ~ N(0,0.02),
no C, bf16 out (seeded synthetic inputs, tensor_core_gemm_02_gb300.workloads).
One step = one gemm_bf16 call on inputs already in HBM.  The metric is
TFLOP/s = 2 M N K / time.  The same line also carries:

  e2e           the same metric through the C ABI with host buffers: each step
                copies A and B from pinned host memory, runs the GEMM and reads
                D back, all inside the timed region (copies of neighbouring
                steps overlap the GEMM on their own streams)
  roofline      the kernel's achieved TFLOP/s against the measured dense bf16
                peak in MEASURED_PEAKS.json (tensor-bound), and the DRAM traffic
                per launch from the committed ncu summary when it is current
  clocks        nvidia-smi samples every 20 ms inside the timed region (median
                SM clock, reasons seen active) and the driver's per-reason
                slowdown counters read at its two ends (reason_us: how long
                each reason held the clocks down in it)
  sustained     the headline GEMM back to back for about 4 s (--sustained-seconds),
                once the power cap has settled, against the measured sustained
                cuBLAS rate (bf16_tflops_sustained)
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample of rows
  variants      the other workloads (f16 1024^3 + C, 8192 x 28672 x 4096 with
                C, the M = 16 skinny case, the gathered 16384-of-65536 rows
                case, scattered rows, the accumulating and FP4-weight skinny
                cases): device time per launch from a CUDA graph of
                back-to-back launches that cycle through copies of the operands
                holding at least twice L2 (no launch finds its inputs in L2),
                with their own roofline (HBM-bound ones against the copy
                bandwidth)

With --impl reference the oracle itself is timed as the comparison arm.

One GPU only.  The library's clustered forms use TMA multicast within one
GPU's memory, and the GEMM has no exchange step to run across GPUs, so the
bench refuses --gpus other than 1 and any launch with WORLD_SIZE > 1.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tensor_core_gemm_02_gb300 import binding, workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
HEADLINE = "bf16_8192"
# dense FP4 (block-scaled) / bf16 and FP8 / bf16 tensor rates: the nominal
# ratios (4.5 and 2.25 PFLOP/s against 2.25), and the ratios one SM's tensor
# pipe shows for one thread issuing 128 x 256 MMAs back to back (kind::mxf4 and
# mxf4nvf4: 32768 flop per clock; kind::mxf8f6f4: 16384; kind::f16: 8192)
FP4_NOMINAL_RATIO, FP4_MEASURED_RATIO = 6.0, 4.0
FP8_NOMINAL_RATIO, FP8_MEASURED_RATIO = 2.0, 2.0
# dense bf16 / f16 tcgen05 rate of one SM: a 128 x N x 16 MMA (2 * 128 * N * 16
# flop) keeps the tensor pipe busy for N / 2 cycles
FLOP_PER_CLK_PER_SM = 8192


# ----------------------------------------------------------------- plumbing

def single_gpu_only(gpus):
    """Exit with a message unless this is one process on one GPU."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if gpus != 1 or world != 1:
        sys.stderr.write(
            f"bench.py runs on one GPU only (--gpus {gpus}, WORLD_SIZE {world}): the "
            "library's clustered forms multicast TMA loads within one GPU's memory and "
            "the GEMM has no step that spans GPUs\n")
        sys.exit(2)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash():
    """Hash of the CUDA sources; a stored ncu traffic figure is used only if it matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_core_gemm_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key):
    """DRAM bytes per launch recorded from an ncu capture of the current sources, or None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash():
        return None
    e = d.get("kernels", {}).get(kernel_key)
    return None if e is None else e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs,
    plus the driver's cumulative per-reason slowdown counters (microseconds) read
    right before and right after it, which catch a reason that was active between
    two samples."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "power.draw.instant")
    COUNTERS = ("sw_power_cap", "sw_thermal_slowdown", "hw_thermal_slowdown",
                "hw_power_brake_slowdown")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def counters(self):
        """The cumulative slowdown counters (us per reason), or None if unavailable."""
        q = ",".join("clocks_event_reasons_counters." + c for c in self.COUNTERS)
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=10)
            vals = [int(x.strip()) for x in out.stdout.strip().split(",")]
        except (OSError, ValueError, subprocess.SubprocessError):
            return None
        return dict(zip(self.COUNTERS, vals)) if len(vals) == len(self.COUNTERS) else None

    def mark(self, which):
        """Host wall-clock bounds of the timed region (samples outside are dropped);
        the slowdown counters are read just before the start and just after the end."""
        if which == "t_start":
            self.c_start = self.counters()
        setattr(self, which, time.time())
        if which == "t_end":
            self.c_end = self.counters()

    def __enter__(self):
        self.t_start = self.t_end = None
        self.c_start = self.c_end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.out.name) == 0:
                time.sleep(0.05)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()

    def summary(self):
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    mask = int(parts[5], 16) if parts[5].startswith("0x") else 0
                    try:
                        inst = float(parts[10]) if len(parts) > 10 else float(parts[4])
                    except ValueError:
                        inst = float(parts[4])
                    rows.append({"t": ts, "sm": float(parts[2]), "max": float(parts[3]),
                                 "power": float(parts[4]), "power_inst": inst, "mask": mask,
                                 "hw_slowdown": parts[6] == "Active",
                                 "hw_thermal_slowdown": parts[7] == "Active",
                                 "sw_thermal_slowdown": parts[8] == "Active",
                                 "sw_power_cap": parts[9] == "Active"})
                except ValueError:
                    continue
        os.unlink(self.out.name)
        if self.t_start is not None and self.t_end is not None:
            inside = [r for r in rows if self.t_start <= r["t"] <= self.t_end]
            if not inside and rows:  # region shorter than the sampling period
                mid = 0.5 * (self.t_start + self.t_end)
                inside = sorted(rows, key=lambda r: abs(r["t"] - mid))[:2]
            rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        pw = sorted(r["power"] for r in rows)
        load = rows
        reasons = {k for r in rows for k in ("hw_slowdown", "hw_thermal_slowdown",
                                             "sw_thermal_slowdown", "sw_power_cap") if r[k]}
        # microseconds each reason held the clocks down inside the timed region
        reason_us = None
        if self.c_start is not None and self.c_end is not None:
            reason_us = {k: self.c_end[k] - self.c_start[k] for k in self.COUNTERS}
            reasons |= {k for k, v in reason_us.items() if v > 0}
        reasons = sorted(reasons)
        # every reason in the active bitmask (nvidia-smi's clocks_event_reasons bits)
        names = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                 0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
        active = sorted({n for r in rows for b, n in names.items() if r["mask"] & b})
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "active_reasons": active, "samples": len(rows), "power_w_max": max(pw),
                "power_instant_w_max": max(r["power_inst"] for r in rows),
                "reason_us": reason_us,
                "window_us": (round((self.t_end - self.t_start) * 1e6)
                              if self.t_start is not None and self.t_end is not None else None),
                "sm_mhz_samples": [r["sm"] for r in rows][:40]}


def kernel_key(plan, p=None):
    """The kernel instance a plan launches for problem p, as ncu names it (for
    profiles/traffic.json): tile_gemm_kernel<BN, STAGES, PAIR, NSUB, MC, MODE, MX>,
    MODE 0 plain, 1 scattered rows, 2 reduce-add, MX the operand kind (0 16-bit,
    1 packed FP4, 2 the 16U4 FP4 image); skinny_gemm_kernel<MP, KBOX, W4, MX>
    (W4 FP4 weights, MX both operands FP4)."""
    mode = 0 if p is None else (1 if p.scatter else (2 if p.accumulate else 0))
    if plan.kernel in (11, 12, 13, 14):  # FP4 operands with block scales (last: operand kind)
        pair = 1 if plan.kernel >= 13 else 0
        return (f"tile_gemm_kernel<{plan.bn}, {plan.stages}, {pair}, 1, 1, 0, "
                f"{1 if plan.kernel in (11, 13) else 2}>")
    if plan.kernel == 15:  # both operands FP4, M <= 64
        return f"skinny_gemm_kernel<{plan.bm}, 1, 0, 1>"
    if plan.kernel == 2:  # (FP4 stages hold four 64-wide K blocks)
        return ("skinny_gemm_kernel<{}, 4, 1, 0>" if p is not None and p.fp4
                else "skinny_gemm_kernel<{}, 1, 0, 0>").format(plan.bm)
    if plan.kernel == 10:
        return "tiny_gemm_kernel"
    form = {3: "256, 6, 1, 1, 1", 4: "256, 4, 1, 2, 1", 7: "256, 4, 1, 2, 2",
            8: "256, 6, 1, 1, 2", 9: "256, 4, 1, 2, 4"}.get(plan.kernel)
    if form is None:
        mc = {5: 4, 6: 8}.get(plan.kernel, 1)
        form = f"{plan.bn}, {plan.stages}, 0, 1, {mc}"
    return f"tile_gemm_kernel<{form}, {mode}, 0>"  # (last: operand kind 0, 16-bit)


def plan_of(p, dev):
    if p.e2m1:
        return binding.gemm_query_plan(
            p.M, p.N, p.K, e2m1=p.image,
            sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)
    return binding.gemm_query_plan(p.M, p.N, p.K, gather=p.idx is not None and not p.scatter,
                                   scatter=p.scatter, fp4=p.fp4,
                                   has_c=p.C is not None and p.beta != 0,
                                   sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)


def launch(p, dev_tensors):
    A, B, C, idx, D = dev_tensors[:5]
    if p.e2m1:
        As, Bs = dev_tensors[5:]
        return binding.gemm_e2m1(A, As, B, Bs, C, D, alpha=p.alpha, beta=p.beta, out=p.out,
                                 image=p.image)
    if p.fp4:
        return binding.gemm_bf16_e2m1(A, B, idx, C, D, alpha=p.alpha, beta=p.beta, out=p.out)
    if p.accumulate:
        return binding.gemm_accumulate(A, B, D, alpha=p.alpha)
    if p.scatter:
        return binding.gemm_scatter_rows(A, B, idx, D, C, alpha=p.alpha, beta=p.beta)
    if idx is not None:
        return binding.gemm_gather_rows(A, idx, B, C, D, alpha=p.alpha, beta=p.beta, out=p.out)
    if A.dtype == torch.bfloat16:
        return binding.gemm_bf16(A, B, C, D, alpha=p.alpha, beta=p.beta, out=p.out)
    return binding.gemm_f16(A, B, C, D, alpha=p.alpha, beta=p.beta, out=p.out)


def to_device(p, dev):
    A = p.A.to(dev)
    B = p.B.to(dev)
    C = p.C.to(dev) if p.C is not None else None
    idx = p.idx.to(dev) if p.idx is not None else None
    if p.fp4:
        idx = p.Bs.to(dev)  # (the scales ride in the index slot)
    if p.accumulate:
        D = p.D0.to(dev).contiguous()
    elif p.scatter:
        D = (p.D0.to(dev) if p.D0 is not None else
             torch.zeros((p.d_rows, p.N), dtype=workloads.OUT_TORCH[p.out], device=dev))
    else:
        D = torch.empty((p.M, p.N), dtype=workloads.OUT_TORCH[p.out], device=dev)
    if p.e2m1:
        return A, B, C, idx, D, p.As.to(dev), p.Bs.to(dev)
    return A, B, C, idx, D


def algorithmic_bytes(p):
    """Bytes the GEMM must move at least once: A (or the gathered rows), B, C, D, idx
    (scattered form: the M rows of C read and of D written; accumulating form: D
    read and written)."""
    if p.e2m1:  # codes and scales of both operands
        a = p.M * p.K // 2 + p.As.numel()
        b = p.N * p.K // 2 + p.Bs.numel()
        c = p.M * p.N * 4 if (p.C is not None and p.beta != 0) else 0
        return a + b + c + p.M * p.N * workloads.OUT_TORCH[p.out].itemsize
    esz = p.A.element_size()
    a = p.M * p.K * esz
    b = p.N * p.K * esz if not p.fp4 else p.N * p.K // 2 + p.Bs.numel()  # FP4: codes + scales
    c = p.M * p.N * 4 if (p.C is not None and p.beta != 0) else 0
    d = p.M * p.N * workloads.OUT_TORCH[p.out].itemsize * (2 if p.accumulate else 1)
    i = p.M * 4 if p.idx is not None else 0
    return a + b + c + d + i


# ----------------------------------------------------------------- our arm

def time_headline(p, dev, steps, warmup):
    tensors = to_device(p, dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        launch(p, tensors)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        torch.cuda.synchronize()
        clocks.mark("t_start")
        e0.record(stream)
        for _ in range(steps):
            launch(p, tensors)
        e1.record(stream)
        torch.cuda.synchronize()
        clocks.mark("t_end")
    ms = e0.elapsed_time(e1)
    status = binding.gemm_check_device_status()
    if status != binding.GEMM_OK:
        raise RuntimeError(f"device status after timing: {binding.gemm_status_string(status)}")
    del tensors
    return ms, clocks.summary()


def time_sustained(p, dev, seconds):
    """The headline GEMM back to back for about `seconds` (batches of 50 launches
    until the host clock passes the mark), timed with CUDA events around the
    whole run, clocks sampled meanwhile: the rate once the power cap has settled,
    to set beside the measured sustained cuBLAS figure."""
    tensors = to_device(p, dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        launch(p, tensors)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = 0
    with ClockSampler(dev.index) as clocks:
        clocks.mark("t_start")
        e0.record(stream)
        t0 = time.time()
        marks = []
        while time.time() - t0 < seconds:
            for _ in range(50):
                launch(p, tensors)
            n += 50
            marks.append(torch.cuda.Event())
            marks[-1].record(stream)
            # keep the host one batch ahead of the device: the queue never runs dry
            if len(marks) > 1:
                marks.pop(0).synchronize()
        e1.record(stream)
        torch.cuda.synchronize()
        clocks.mark("t_end")
    ms = e0.elapsed_time(e1)
    status = binding.gemm_check_device_status()
    if status != binding.GEMM_OK:
        raise RuntimeError(f"device status after the sustained run: {binding.gemm_status_string(status)}")
    del tensors
    return ms, n, clocks.summary()


def time_e2e(p, dev, steps):
    """Host buffers through the C ABI, pipelined over three streams.

    Every step copies its A and B from pinned host memory (H2D), runs the GEMM
    and copies its D back to pinned host memory (D2H), all inside the timed
    region.  Two sets of device buffers let step i+1's H2D and step i-1's D2H
    run on their own streams while step i computes, as a host-fed pipeline
    would; a step waits only for the copies and GEMM it depends on.
    """
    A_h = p.A.pin_memory()
    B_h = p.B.pin_memory()
    D_h = [torch.empty((p.M, p.N), dtype=workloads.OUT_TORCH[p.out]).pin_memory()
           for _ in range(2)]
    A_d = [torch.empty_like(A_h, device=dev) for _ in range(2)]
    B_d = [torch.empty_like(B_h, device=dev) for _ in range(2)]
    D_d = [torch.empty_like(D_h[0], device=dev) for _ in range(2)]
    s_in, s_mm, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        ev_in = [None, None]
        ev_mm = [None, None]
        ev_out = [None, None]
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if ev_mm[b] is not None:
                    s_in.wait_event(ev_mm[b])  # the GEMM two steps back is done with buffer b
                A_d[b].copy_(A_h, non_blocking=True)
                B_d[b].copy_(B_h, non_blocking=True)
                ev_in[b] = torch.cuda.Event()
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_mm):
                s_mm.wait_event(ev_in[b])
                if ev_out[b] is not None:
                    s_mm.wait_event(ev_out[b])  # D of two steps back has been read out
                binding.gemm_bf16(A_d[b], B_d[b], None, D_d[b], alpha=p.alpha, beta=p.beta,
                                  out=p.out, stream=s_mm)
                ev_mm[b] = torch.cuda.Event()
                ev_mm[b].record(s_mm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mm[b])
                D_h[b].copy_(D_d[b], non_blocking=True)
                ev_out[b] = torch.cuda.Event()
                ev_out[b].record(s_out)

    run(2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    h2d = A_h.numel() * A_h.element_size() + B_h.numel() * B_h.element_size()
    d2h = D_h[0].numel() * D_h[0].element_size()
    return ms, h2d, d2h


def set_bytes(tensors):
    """Device bytes of one launch's operands (inputs and output)."""
    return sum(t.numel() * t.element_size() for t in tensors if t is not None)


def time_variant(name, dev, reps, flush=None):
    """Device time per launch, without host launch gaps: a CUDA graph of back-to-back
    launches, replayed and timed with events on its stream.  Operands smaller than
    twice L2 are replicated so that the launches cycle through copies holding at
    least twice L2 together: no launch finds its inputs in L2 from an earlier one
    (a copy's data was last touched at least an L2's worth of traffic before)."""
    p = workloads.WORKLOADS[name]()
    first = to_device(p, dev)
    one = set_bytes(first)
    copies = 1 if one >= 2 * L2_BYTES else -(-2 * L2_BYTES // one)
    copies = max(1, min(copies, (6 << 30) // max(one, 1)))
    sets = [first] + [to_device(p, dev) for _ in range(copies - 1)]
    n = -(-max(reps, copies) // copies) * copies
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for t in sets:
            launch(p, t)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(n):
            launch(p, sets[i % copies])
    times = []
    with torch.cuda.stream(stream):  # (a graph replays on the current stream)
        graph.replay()
        torch.cuda.synchronize()
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) / n)
    status = binding.gemm_check_device_status()
    if status != binding.GEMM_OK:
        raise RuntimeError(f"{name}: device status {binding.gemm_status_string(status)}")
    ms = statistics.median(times)
    plan = plan_of(p, dev)
    del graph, sets, first
    torch.cuda.empty_cache()
    return p, ms, plan, (f"CUDA graph of {n} back-to-back launches cycling through {copies} "
                         f"cop{'y' if copies == 1 else 'ies'} of the operands "
                         f"({copies * one / 1e6:.0f} MB, >= 2x L2 when copied); median of 5 replays")


def oracle_rows_rate(p, seconds, threads):
    """Run the oracle on whole output rows for about `seconds`; returns (flops/s, rows)."""
    import oracle

    rows = threads  # calibration: one row per thread
    t0 = time.time()
    oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta, idx=p.idx, threads=threads, rows=(0, rows))
    dt = max(time.time() - t0, 1e-3)
    rows = int(max(1, min(p.M, (seconds / dt) * rows)))
    # whole multiples of the thread count keep every host core busy
    rows = max(threads, (rows // threads) * threads) if p.M >= threads else rows
    rows = min(rows, p.M)
    t0 = time.time()
    oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta, idx=p.idx, threads=threads, rows=(0, rows))
    dt = time.time() - t0
    return 2.0 * rows * p.N * p.K / dt, rows, dt


# NVIDIA's published dense (no 2:4 sparsity) bf16 / fp16 tensor figure for one GB300
NOMINAL_DENSE_BF16_TFLOPS = 2250.0


def spec_peak(sms, clocks, achieved):
    """The chip's dense bf16 tensor peak: NVIDIA's published dense figure, and
    from its SM count, the per-SM rate and the SM clock at the maximum clock and
    at the median clock sampled during the timed region, with the achieved rate
    (TFLOP/s) as a fraction of each."""
    out = {"flop_per_clk_per_sm": FLOP_PER_CLK_PER_SM, "sms": sms,
           "source": "one SM's tensor pipe runs a 128 x N x 16 bf16 MMA in N/2 cycles "
                     "(8192 flop per clock); x SMs x SM clock",
           "nominal_dense_tflops": NOMINAL_DENSE_BF16_TFLOPS,
           "frac_of_nominal": round(achieved / NOMINAL_DENSE_BF16_TFLOPS, 4)}
    for key, mhz in (("max", clocks.get("sm_max_mhz")), ("median", clocks.get("sm_mhz"))):
        if mhz:
            peak = FLOP_PER_CLK_PER_SM * sms * mhz * 1e6 / 1e12
            out[f"{key}_mhz"] = mhz
            out[f"peak_at_{key}_mhz"] = round(peak, 1)
            out[f"frac_at_{key}_mhz"] = round(achieved / peak, 4)
    return out


def run_ours(args):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load_library()
    peaks = measured_peaks()

    p = workloads.WORKLOADS[HEADLINE]()
    flops = p.flops
    ms_total, clocks = time_headline(p, dev, args.steps, args.warmup)
    ms_step = ms_total / args.steps
    value = flops / (ms_step * 1e-3) / 1e12
    achieved = value

    e2e_steps = min(args.steps, 20)
    e2e_ms, h2d, d2h = time_e2e(p, dev, e2e_steps)
    sustained = None
    if args.sustained_seconds > 0:
        s_ms, s_n, s_clocks = time_sustained(p, dev, args.sustained_seconds)
        s_rate = s_n * flops / (s_ms * 1e-3) / 1e12
        s_peak = peaks.get("bf16_tflops_sustained")
        sustained = {"value": round(s_rate, 2), "unit": "TFLOP/s", "launches": s_n,
                     "seconds": round(s_ms * 1e-3, 3), "peak": s_peak,
                     "frac": round(s_rate / s_peak, 4) if s_peak else None,
                     "peak_source": f"{peaks['source']} bf16_tflops_sustained (cuBLAS, 4 s)",
                     "clocks": {k: s_clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons",
                                                              "reason_us", "window_us",
                                                              "power_instant_w_max")}}

    result = {
        "metric": "GEMM TFLOP/s (bf16 8192^3, bf16 out)",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) / N(0,0.02) bf16)",
        "config": {"workload": "bf16 GEMM M=N=K=8192, A~N(0,1), B~N(0,0.02), C=0, bf16 out",
                   "M": 8192, "N": 8192, "K": 8192, "parallelism": "one GPU",
                   "l2": "inputs larger than L2 (A+B = 256 MiB > 129 MB)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": round(e2e_ms, 4),
                "how": "pinned host A, B -> device, gemm_bf16, D -> pinned host, every step; "
                       "copies of neighbouring steps overlap on their own streams; "
                       "host wall clock over all steps"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "peak_source": f"{peaks['source']} bf16_tflops (burst)",
                     "traffic": stored_traffic(f"{kernel_key(plan_of(p, dev), p)}@{HEADLINE}"),
                     "kernel": kernel_key(plan_of(p, dev), p),
                     "algorithmic_flops_per_launch": flops,
                     "chip_dense_bf16_peak": spec_peak(
                         torch.cuda.get_device_properties(dev).multi_processor_count,
                         clocks, achieved)},
    }
    if sustained is not None:
        result["sustained"] = sustained

    if args.variants:
        variants = {}
        for name in ("f16_1024", "mlp_8192x28672x4096", "skinny_16x28672x4096",
                     "gather_16384_of_65536", "scatter_16384_into_65536",
                     "skinny_accumulate_16x28672x4096", "fp4_skinny_16x28672x4096",
                     "e2m1_16x28672x4096", "e2m1_8192"):
            vp, ms, plan, how = time_variant(name, dev, args.variant_reps)
            tflops = vp.flops / (ms * 1e-3) / 1e12
            gbs = algorithmic_bytes(vp) / (ms * 1e-3) / 1e9
            hbm_bound = name in ("skinny_16x28672x4096", "skinny_accumulate_16x28672x4096",
                                 "fp4_skinny_16x28672x4096", "e2m1_16x28672x4096")
            # the tensor peak of the variant's operand kind (FP4: block-scaled MMAs)
            if vp.e2m1:
                nominal = FP4_NOMINAL_RATIO if vp.image == 0 else FP8_NOMINAL_RATIO
                measured = FP4_MEASURED_RATIO if vp.image == 0 else FP8_MEASURED_RATIO
            else:
                nominal = measured = 1.0
            t_peak = peaks["bf16_tflops"] * nominal
            variants[name] = {
                "ms": round(ms, 5), "TFLOP/s": round(tflops, 2), "GB/s": round(gbs, 1),
                "algorithmic_bytes": algorithmic_bytes(vp),
                "kernel": {1: "tile (single CTA)", 2: "skinny (swap-AB, stream-K)",
                           11: "tile (single CTA, FP4 block-scaled, kind::mxf4)",
                           12: "tile (single CTA, FP4 block-scaled, kind::mxf8f6f4)",
                           15: "skinny (swap-AB, stream-K, FP4 block-scaled, kind::mxf4)",
                           3: "tile (CTA pair)", 4: "tile (CTA pair, two N halves)",
                           5: "tile (4-CTA cluster, A multicast)",
                           6: "tile (8-CTA cluster, A multicast)",
                           7: "tile (two CTA pairs, 256 x 512, A multicast)",
                           8: "tile (two CTA pairs, 256 x 256, A multicast)",
                           9: "tile (four CTA pairs, 256 x 512, A multicast)"}[plan.kernel],
                "tile": f"{plan.bm}x{plan.bn}", "grid": plan.grid, "splits": plan.splits,
                "roofline": dict(({"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
                                  if hbm_bound else
                                  {"bound": "tensor", "achieved": round(tflops, 2),
                                   "peak": round(t_peak, 1), "unit": "TFLOP/s",
                                   "frac": round(tflops / t_peak, 4),
                                   **({"peak_source": f"measured bf16 x {nominal:g} (nominal "
                                                      f"ratio); x {measured:g} (per-SM MMA rate "
                                                      f"measured): {peaks['bf16_tflops'] * measured:.1f}",
                                       "frac_of_measured_mma_rate":
                                           round(tflops / (peaks["bf16_tflops"] * measured), 4)}
                                      if vp.e2m1 else {})}),
                                 traffic=stored_traffic(f"{kernel_key(plan, vp)}@{name}"),
                                 kernel=kernel_key(plan, vp)),
                "timing": how,
            }
        result["variants"] = variants

    threads = len(os.sched_getaffinity(0))
    rate, rows, dt = oracle_rows_rate(p, args.cpu_seconds, threads)
    result["cpu_baseline"] = {"value": round(rate / 1e12, 6), "unit": "TFLOP/s",
                              "cores": threads, "kind": "oracle",
                              "sample": f"{rows} full output rows of the 8192^3 bf16 GEMM "
                                        f"(fp64 oracle, {dt:.1f} s)"}
    print(json.dumps(result), flush=True)


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle as the comparison arm: each step computes a bounded sample of rows."""
    p = workloads.WORKLOADS[HEADLINE]()
    threads = len(os.sched_getaffinity(0))
    import oracle
    oracle.load()
    # size each step so that warm-up plus timed steps take about two minutes
    t0 = time.time()
    oracle.gemm(p.A, p.B, None, 1.0, 0.0, threads=threads, rows=(0, threads))
    per_row = max(time.time() - t0, 1e-3) / threads
    budget = 120.0 / (args.steps + args.warmup)
    rows = int(max(1, min(p.M // 2, budget / per_row)))
    for _ in range(args.warmup):
        oracle.gemm(p.A, p.B, None, 1.0, 0.0, threads=threads, rows=(0, rows))
    t0 = time.time()
    for s in range(args.steps):
        r0 = (s * rows) % (p.M - rows)
        oracle.gemm(p.A, p.B, None, 1.0, 0.0, threads=threads, rows=(r0, r0 + rows))
    dt = (time.time() - t0) / args.steps
    value = 2.0 * rows * p.N * p.K / dt / 1e12
    print(json.dumps({
        "impl": "reference",
        "metric": "GEMM TFLOP/s (bf16 8192^3, bf16 out)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "bf16 GEMM M=N=K=8192, A~N(0,1), B~N(0,0.02), C=0, bf16 out",
                   "M": 8192, "N": 8192, "K": 8192},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{rows} full output rows per step (fp64 oracle)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_case(args):
    """Run one workload's GEMM warmup + steps times and exit (a target for profilers)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p = workloads.WORKLOADS[args.case]()
    tensors = to_device(p, dev)
    for _ in range(args.warmup + args.steps):
        launch(p, tensors)
    torch.cuda.synchronize()
    status = binding.gemm_check_device_status()
    if status != binding.GEMM_OK:
        raise RuntimeError(f"device status {binding.gemm_status_string(status)}")
    print(f"case {args.case}: {args.warmup} + {args.steps} launches ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-variants", dest="variants", action="store_false")
    ap.add_argument("--variant-reps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--sustained-seconds", type=float, default=4.0,
                    help="length of the back-to-back sustained leg (0: skip it)")
    ap.add_argument("--case", choices=sorted(workloads.WORKLOADS), default=None,
                    help="only launch this workload's GEMM warmup + steps times (profiling)")
    args = ap.parse_args()
    single_gpu_only(args.gpus)
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
