#!/usr/bin/env python3
"""Benchmark of the causal linear-attention training step on GB300.

One step = one causal forward (la_causal_fwd) plus one causal backward
(la_causal_bwd) through the C ABI over a batch of B=4 sequences x H=8 heads of
N=3072 tokens with D=M=64, bf16 in and out, fp32 accumulation (the 32x32x3
autoregressive-image workload of "Transformers are RNNs").  Inputs are seeded
N(0, 1) draws, resident in HBM before the timed region; L2 is flushed (a
256 MiB write) before every timed step, outside the step's events.

Prints one JSON line.  `value` is tokens/s = B*N / (device time of one step),
summed over ranks (independent replicas, weak scaling).  Extra objects:
  roofline      the dominant call (la_causal_bwd), algorithmic bytes per call /
                its live CUDA-event duration, against the measured HBM copy rate
  cpu_baseline  the fp64 CPU oracle (recurrent form, fwd+bwd) on the host cores
  e2e           the same step with pinned host buffers and the copies inside
  secondary     non-causal fwd+bwd, prefill, decode-step and projected
                decode-step measurements
  clocks        nvidia-smi samples taken during the timed region

`--impl reference` times the CPU oracle itself (rank 0 only) on the same
workload, one bounded sample per step.

Multi-GPU (torchrun, one process per GPU): every rank runs the same workload
on its own GPU; there is no collective on the data path (the sequences are
independent); timing is the max over ranks between barriers.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal linear-attn fwd+bwd tokens/s (N=3072, D=M=64) and % of roofline"
WORKLOAD = "causal_cifar_bf16"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="skip the non-causal/decode lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--secondary-only", action="store_true",
                    help="run only the secondary measurements (one JSON object); for profiling "
                         "those kernels")
    ap.add_argument("--only", default=None,
                    help="with --secondary-only: a comma-separated subset of " + ", ".join(SECONDARY))
    ap.add_argument("--sweep", action="store_true",
                    help="sequence-length sweep N = 2^9 .. 2^16 with B * N fixed: causal fwd+bwd "
                         "time and peak allocated memory per sample (one JSON object)")
    return ap.parse_args()


# ------------------------------------------------------------------ plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend, rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons, n = [], None, set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": n}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (read-only queries,
    ctypes on the driver's libnvidia-ml), one sample per call of sample():
    time_calls takes one per timed step, right after the step's L2 flush is
    enqueued, so the samples cover the timed region at any step count."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, dev):
        import ctypes
        self.ok, self.sm, self.reasons = False, [], 0
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            bus = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
            dom = getattr(torch.cuda.get_device_properties(dev), "pci_domain_id", 0)
            dv = getattr(torch.cuda.get_device_properties(dev), "pci_device_id", 0)
            rc = 1
            if bus is not None:
                rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(
                    f"{dom:08x}:{bus:02x}:{dv:02x}.0".encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.lib.nvmlDeviceGetHandleByIndex_v2(dev.index or 0, ctypes.byref(self.h))
            if rc != 0:
                return
            self.ct = ctypes
            self.val = ctypes.c_uint()
            self.rs = ctypes.c_ulonglong()
            self.max_mhz = None
            if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(self.val)) == 0:
                self.max_mhz = float(self.val.value)
            self.get_reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def sample(self):
        if not self.ok:
            return
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(self.val)) == 0:
            self.sm.append(float(self.val.value))
        if self.get_reasons(self.h, self.ct.byref(self.rs)) == 0:
            self.reasons |= int(self.rs.value)

    def summary(self, ms_per_step):
        if not self.ok or not self.sm:
            return None
        med = statistics.median(self.sm)
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.reasons & b),
                "samples": len(self.sm), "sm_mhz_min": min(self.sm),
                "source": "NVML, one sample per timed step",
                "ms_x_mhz": round(ms_per_step * med, 3)}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip() + f" ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# the files the timed causal tcgen05 kernels are built from
CAUSAL_TC_SOURCES = ("causal_tc.cu", "causal_tc_bwd.cu", "tc.cuh", "tc_chunk.cuh", "common.cuh")


def kernel_source_hash():
    """Hash of the causal tcgen05 kernels' sources, to tell whether stored ncu
    counters still describe the kernels being timed."""
    csrc = os.path.join(ROOT, "kernelized_causal_attention_gb300", "csrc")
    h = hashlib.sha256()
    for name in CAUSAL_TC_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key):
    """DRAM bytes per call from the committed ncu summary, or None when the
    kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except (OSError, ValueError):
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("per_call_dram_bytes", {}).get(kernel_key)


# ------------------------------------------------------------- byte counting

def causal_bytes(B, H, N, D, M, elt):
    """Algorithmic bytes per call (recurrence form: every input read once and
    every output written once)."""
    th = B * H * N
    fwd = th * (elt * (2 * D + M) + elt * M + 4)                   # q,k,v in; out, den out
    bwd = th * (elt * (2 * D + M) + 2 * elt * M + 4 + elt * (2 * D + M))  # q,k,v,out,dout,den; dq,dk,dv
    return fwd, bwd


# ------------------------------------------------------------------ our arm

LEAD_CYCLES = 200_000  # about 100 us of GPU idle after each flush, untimed


def lead(torch):
    """Keeps the GPU busy (untimed) for about 100 us after the L2 flush, so
    that the host has enqueued the whole step before the step's first event
    is reached: the device time then excludes host-side launch overhead (that
    overhead is part of the e2e figure instead)."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(LEAD_CYCLES)


def time_calls(fns, steps, flush, torch, dist, dev, with_median=False, sample=None, split=True):
    """Runs `steps` iterations of the call sequence `fns`, with an L2 flush
    before each; returns per-call mean ms (None unless split) and per-step
    mean ms (device time), and with_median the per-step median ms as well.

    With split an event follows every call.  An event between two calls ends
    the overlap that programmatic dependent launch gives the second call's
    first kernel with the first call's last one (its CTAs start and run their
    prologue while the other drains), so a step is timed without them: events
    at the step's start and end only."""
    n = len(fns)
    ne = n + 1 if split else 2
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ne)] for _ in range(steps)]
    for i in range(steps):
        flush()
        if sample is not None:
            sample()  # the GPU is busy with the flush meanwhile
        lead(torch)
        ev[i][0].record()
        for j, fn in enumerate(fns):
            fn()
            if split:
                ev[i][j + 1].record()
        if not split:
            ev[i][1].record()
    torch.cuda.synchronize()
    per_call = ([statistics.fmean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
                 for j in range(n)] if split else None)
    steps_ms = [ev[i][0].elapsed_time(ev[i][ne - 1]) for i in range(steps)]
    if with_median:
        return per_call, statistics.fmean(steps_ms), statistics.median(steps_ms)
    return per_call, statistics.fmean(steps_ms)


def step_and_calls(fns, steps, flush, torch, dev):
    """(per-call mean ms from a pass with an event after each call, step mean
    ms from a pass with events at the step boundaries only)."""
    per_call, _ = time_calls(fns, steps, flush, torch, None, dev)
    _, ms = time_calls(fns, steps, flush, torch, None, dev, split=False)
    return per_call, ms


def run_ours(args, dist):
    import torch

    import kernelized_causal_attention_gb300 as la
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    dist.init("nccl" if dist.world > 1 else "gloo")
    la.lib()
    w = WORKLOADS[WORKLOAD]
    B, H, N, D, M = w.B, w.H, w.N, w.D, w.M
    dt = la.LA_BF16
    q, k, v, g = causal_inputs(B, H, N, D, M, w.dtype, w.seed + dist.rank * 1000)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty(B, H, N, M, dtype=torch.bfloat16, device=dev)
    den = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wsf = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, dev)
    wsb = la.workspace(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, dt, dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.zero_()

    fwd = lambda: la.la_causal_fwd(qd, kd, vd, out, den, wsf, B, H, N, D, M, dt)
    bwd = lambda: la.la_causal_bwd(qd, kd, vd, out, den, gd, dq, dk, dv, wsb, B, H, N, D, M, dt)

    for _ in range(max(3, args.warmup)):
        flush()
        fwd()
        bwd()
    torch.cuda.synchronize()

    nv = NvmlClocks(torch, dev)
    clocks = ClockSampler(dist.local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _, ms_step, ms_median = time_calls([fwd, bwd], args.steps, flush, torch, dist, dev,
                                       with_median=True, sample=nv.sample, split=False)
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t0
    smi = clocks.stop()
    clk = nv.summary(ms_step) or dict(smi)
    clk["nvidia_smi"] = smi  # 100 ms samples over the same window (few or none for short runs)
    # outside the timed region: the per-call times (a second pass of as many
    # steps with an event after each call, which serialises the two calls)
    # and the same step with L2 left warm (inputs partly resident)
    (ms_fwd, ms_bwd), ms_split = time_calls([fwd, bwd], args.steps, flush, torch, dist, dev)
    _, ms_warm = time_calls([fwd, bwd], 200, lambda: None, torch, dist, dev, split=False)

    ms_step_max = dist.max(ms_step, dev)
    ms_bwd_max = dist.max(ms_bwd, dev)
    ms_fwd_max = dist.max(ms_fwd, dev)
    tokens = B * N
    value = dist.world * tokens / (ms_step_max / 1e3)
    launches = args.steps * (la.la_kernel_launches(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt)
                             + la.la_kernel_launches(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, dt))

    peaks = measured_peaks()
    fwd_b, bwd_b = causal_bytes(B, H, N, D, M, 2)
    achieved = bwd_b / (ms_bwd_max / 1e3) / 1e9
    traffic = stored_traffic("la_causal_bwd")
    roofline = {"bound": "hbm", "kernel": "la_causal_bwd", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "alg_bytes": bwd_b, "ms": round(ms_bwd_max, 5),
                "peak_source": peaks["source"]}
    step_alg = (fwd_b + bwd_b) / (ms_step_max / 1e3) / 1e9
    step_roof = {"alg_bytes": fwd_b + bwd_b, "achieved_gbs": round(step_alg, 1),
                 "frac": round(step_alg / peaks["hbm_gbs"], 4), "fwd_ms": round(ms_fwd_max, 5),
                 "fwd_gbs": round(fwd_b / (ms_fwd_max / 1e3) / 1e9, 1),
                 "split_step_ms": round(dist.max(ms_split, dev), 5),
                 "per_call_timing": "fwd_ms and the roofline's ms come from a second pass with an "
                                    "event after each call; that event keeps the backward's first "
                                    "kernel from overlapping the forward's last (split_step_ms)"}

    e2e = measure_e2e(la, torch, dev, q, k, v, g, out, den, wsf, wsb, B, H, N, D, M, dt,
                      max(3, min(args.steps, 200)), flush, dist)

    res = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic",
           "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "D": D, "M": M,
                      "in_dtype": "bf16", "accumulate": "fp32", "global_batch": B * dist.world,
                      "seq_len": N, "parallelism": f"replicas{dist.world}",
                      "l2": "flushed before every timed step (256 MiB write, untimed)",
                      "enqueue": "GPU idles ~100 us after each flush (untimed) so the host enqueues the step ahead",
                      "timing": "CUDA events at each step's start and end (none between the calls)"},
           "roofline": roofline, "step_roofline": step_roof, "e2e": e2e,
           "gpu_launches": launches, "clocks": clk, "wall_s_timed_region": round(wall, 3),
           "median_ms_per_step": round(dist.max(ms_median, dev), 5),
           "warm": {"ms_per_step": round(dist.max(ms_warm, dev), 5),
                    "value": round(dist.world * tokens / (dist.max(ms_warm, dev) / 1e3), 1),
                    "steps": 200, "l2": "not flushed between steps"}}
    if not args.no_secondary:
        res["secondary"] = secondary(la, torch, dev, flush, peaks,
                                     with_cpu=dist.rank == 0 and not args.no_cpu)
    la.check_device_status()  # raises if a bounded wait inside a kernel ran out
    if dist.rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(q, k, v, g, B, H, N)
    dist.close()
    return res


def measure_e2e(la, torch, dev, q, k, v, g, out, den, wsf, wsb, B, H, N, D, M, dt, steps, flush,
                dist):
    """The step through the public API with pinned host inputs and results:
    every step copies its q, k, v, dout host -> device, runs both calls and
    copies dq, dk, dv device -> host, all inside the timed region.

    Steps are pipelined the way a training loop would run them: a copy-in
    stream, the compute stream and a copy-out stream, two sets of device
    buffers, and events so that step s's input copy overlaps step s-1's
    calls and step s-2's result copy.  The timed region runs from before the
    first step's input copy to the end of the last step's result copy.  The
    same steps on one stream, copies and calls back to back, are reported as
    `serial_ms_per_step`."""
    hq, hk, hv, hg = (t.pin_memory() for t in (q, k, v, g))
    dq_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    dk_h = torch.empty(k.shape, dtype=k.dtype).pin_memory()
    dv_h = torch.empty(v.shape, dtype=v.dtype).pin_memory()
    sets = []
    for _ in range(2):
        ins = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v, g)]
        outs = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v)]
        sets.append((ins, outs))
    s_in, s_c, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]
    c_done = [ev(), ev()]
    out_done = [ev(), ev()]

    def calls(ins, outs):
        qd, kd, vd, gd = ins
        dq_, dk_, dv_ = outs
        la.la_causal_fwd(qd, kd, vd, out, den, wsf, B, H, N, D, M, dt)
        la.la_causal_bwd(qd, kd, vd, out, den, gd, dq_, dk_, dv_, wsb, B, H, N, D, M, dt)

    def copy_in(ins):
        for d, h in zip(ins, (hq, hk, hv, hg)):
            d.copy_(h, non_blocking=True)

    def copy_out(outs):
        for h, d in zip((dq_h, dk_h, dv_h), outs):
            h.copy_(d, non_blocking=True)

    def pipelined(n):
        for s in range(n):
            b = s % 2
            ins, outs = sets[b]
            with torch.cuda.stream(s_in):
                if s >= 2:
                    s_in.wait_event(c_done[b])  # step s-2 is done reading these inputs
                copy_in(ins)
                in_done[b].record(s_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(in_done[b])
                if s >= 2:
                    s_c.wait_event(out_done[b])  # step s-2's results have left these buffers
                calls(ins, outs)
                c_done[b].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(c_done[b])
                copy_out(outs)
                out_done[b].record(s_out)

    def serial():
        ins, outs = sets[0]
        copy_in(ins)
        calls(ins, outs)
        copy_out(outs)

    torch.cuda.synchronize()
    pipelined(4)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    pipelined(steps)
    s_out.wait_stream(s_c)
    s_out.wait_stream(s_in)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1) / steps, dev)

    for _ in range(3):
        serial()
    torch.cuda.synchronize()
    _, ms_serial = time_calls([serial], steps, flush, torch, dist, dev)
    ms_serial = dist.max(ms_serial, dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg))
    d2h = sum(t.numel() * t.element_size() for t in (dq_h, dk_h, dv_h))
    return {"value": round(dist.world * B * N / (ms / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "steps pipelined over copy-in, compute and copy-out streams (two buffer "
                      "sets); every step's copies inside the timed region",
            "serial_ms_per_step": round(ms_serial, 5)}


def secondary(la, torch, dev, flush, peaks, with_cpu=True, only=None):
    """The 784-token causal fwd+bwd, non-causal fwd+bwd (long speech-like
    sequences with padding), the prefill (causal forward from a state), the
    decode step (256 and 2048 streams x 8 heads), the projected decode step
    (256 and 10,000 streams), each against its roofline, and (with_cpu) the
    fp64 oracle timed beside each on the host cores; then a short
    sequence-length sweep."""
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs, noncausal_inputs
    res = {}
    want = lambda name: only is None or name in only
    # the 784-token (28 x 28) image workload: causal fwd + bwd
    for name in ("causal_mnist_bf16", "causal_cifar_d32_bf16", "causal_cifar_f32"):
        if want(name):
            _causal_line(la, torch, dev, flush, peaks, with_cpu, res, name)
    if want("causal_decay_bf16"):
        _causal_decay(la, torch, dev, flush, peaks, with_cpu, res)
    if want("causal_poly_bf16"):
        _causal_poly(la, torch, dev, flush, peaks, with_cpu, res)
    if want("noncausal_speech_f32"):
        _noncausal(la, torch, dev, flush, peaks, with_cpu, res)
    if want("prefill_cifar_bf16"):
        _prefill(la, torch, dev, flush, peaks, with_cpu, res)
    if want("decode_f32"):
        _decode(la, torch, dev, peaks, with_cpu, res)
    for name in ("decode_proj_bf16", "decode_proj_mnist_bf16"):
        if want(name):
            _decode_proj(la, torch, dev, flush, peaks, with_cpu, res, name)
    # a short sequence-length sweep (the full one is --sweep)
    if want("sweep_causal_bf16"):
        res["sweep_causal_bf16"] = {
            "what": "causal fwd+bwd, B * N = 2^16, H = 8, D = M = 64, bf16, 10 L2-flushed steps a point",
            "points": sweep_points(la, torch, dev, flush, peaks, [1 << 10, 1 << 12, 1 << 14, 1 << 16], 10)}
    if with_cpu:
        model = cpu_model()
        for v in res.values():
            if isinstance(v, dict) and "cpu_baseline" in v:
                v["cpu_baseline"].setdefault("cpu_model", model)
    return res


SECONDARY = ("causal_mnist_bf16", "causal_cifar_d32_bf16", "causal_cifar_f32", "causal_decay_bf16", "causal_poly_bf16", "noncausal_speech_f32", "prefill_cifar_bf16", "decode_f32",
             "decode_proj_bf16", "decode_proj_mnist_bf16", "sweep_causal_bf16")


def _causal_line(la, torch, dev, flush, peaks, with_cpu, res, name):
    """Causal fwd + bwd on a named workload (the 784-token images; the
    3072-token images with the pages' 32-wide heads, or with fp32 inputs)."""
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs
    wm = WORKLOADS[name]
    B, H, N, D, M = wm.B, wm.H, wm.N, wm.D, wm.M
    dt, elt = (la.LA_BF16, 2) if wm.dtype == "bf16" else (la.LA_F32, 4)
    q, k, v, g = causal_inputs(B, H, N, D, M, wm.dtype, wm.seed)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty_like(vd)
    den = torch.empty(B, H, N, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wf = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, dev)
    wb = la.workspace(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, dt, dev)
    fwd = lambda: la.la_causal_fwd(qd, kd, vd, out, den, wf, B, H, N, D, M, dt)
    bwd = lambda: la.la_causal_bwd(qd, kd, vd, out, den, gd, dq, dk, dv, wb, B, H, N, D, M, dt)
    for _ in range(3):
        fwd()
        bwd()
    (mf, mb), ms = step_and_calls([fwd, bwd], 100, flush, torch, dev)
    fb, bb = causal_bytes(B, H, N, D, M, elt)
    gbs = (fb + bb) / (ms / 1e3) / 1e9
    res[name] = {
        "value": round(B * N / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "fwd_ms": round(mf, 5), "bwd_ms": round(mb, 5), "B": B, "H": H, "N": N, "D": D, "M": M,
        "dtype": wm.dtype,
        "path": "tcgen05" if dt == la.LA_BF16 else "CUDA cores (fp32 FFMA)",
        "launches": la.la_kernel_launches(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt)
        + la.la_kernel_launches(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, dt),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": fb + bb,
                     "bytes_per_token_head": (fb + bb) // (B * H * N)},
        "timing": "CUDA events, L2 flushed before each step (100 steps)"}
    if with_cpu:
        res[name]["cpu_baseline"] = cpu_baseline(q, k, v, g, B, H, N, budget_s=5.0)


def _causal_decay(la, torch, dev, flush, peaks, with_cpu, res, gamma=0.99):
    """Causal fwd + bwd with the RetNet decay gamma on the 3072-token image
    workload (the same 1544 bytes per token-head as the undecayed step)."""
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs
    w = WORKLOADS["causal_cifar_bf16"]
    B, H, N, D, M = w.B, w.H, w.N, w.D, w.M
    q, k, v, g = causal_inputs(B, H, N, D, M, w.dtype, w.seed)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty_like(vd)
    den = torch.empty(B, H, N, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wf = la.workspace(la.LA_OP_CAUSAL_FWD_DECAY, B, H, N, D, M, 1, dev)
    wb = la.workspace(la.LA_OP_CAUSAL_BWD_DECAY, B, H, N, D, M, 1, dev)
    fwd = lambda: la.la_causal_fwd_decay(qd, kd, vd, out, den, gamma, wf, B, H, N, D, M, 1)
    bwd = lambda: la.la_causal_bwd_decay(qd, kd, vd, out, den, gd, dq, dk, dv, gamma, wb, B, H, N, D,
                                         M, 1)
    for _ in range(3):
        fwd()
        bwd()
    (mf, mb), ms = step_and_calls([fwd, bwd], 50, flush, torch, dev)
    fb, bb = causal_bytes(B, H, N, D, M, 2)
    gbs = (fb + bb) / (ms / 1e3) / 1e9
    res["causal_decay_bf16"] = {
        "value": round(B * N / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "fwd_ms": round(mf, 5), "bwd_ms": round(mb, 5), "gamma": gamma,
        "B": B, "H": H, "N": N, "D": D, "M": M,
        "launches": la.la_kernel_launches(la.LA_OP_CAUSAL_FWD_DECAY, B, H, N, D, M, 1)
        + la.la_kernel_launches(la.LA_OP_CAUSAL_BWD_DECAY, B, H, N, D, M, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": fb + bb},
        "timing": "CUDA events, L2 flushed before each step (50 steps)"}
    if with_cpu:
        import oracle
        cores = _cores(oracle)
        q1, k1, v1, g1 = (t[:1] for t in (q, k, v, g))  # one batch entry: H sequences
        t0 = time.perf_counter()
        oracle.causal_fwd(q1, k1, v1, "recurrent", nthreads=cores, gamma=gamma)
        oracle.causal_bwd(q1, k1, v1, g1, "recurrent", nthreads=cores, gamma=gamma)
        el = time.perf_counter() - t0
        res["causal_decay_bf16"]["cpu_baseline"] = {
            "value": round(N / el, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one batch entry (H={H} sequences of N={N}), fwd+bwd recurrent form, {el:.2f} s"}


def _causal_poly(la, torch, dev, flush, peaks, with_cpu, res):
    """Causal fwd + bwd with the degree-2 polynomial kernel sim = (q . k)^2 on
    the 3072-token shape with 8-wide heads (36 features): q, k, v, out, den
    in and out once, 872 bytes per token-head."""
    from kernelized_causal_attention_gb300.workloads import causal_inputs
    B, H, N, D, M = 4, 8, 3072, 8, 64
    q, k, v, g = causal_inputs(B, H, N, D, M, "bf16", 12)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty_like(vd)
    den = torch.empty(B, H, N, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wf = la.workspace(la.LA_OP_CAUSAL_FWD_POLY, B, H, N, D, M, 1, dev)
    wb = la.workspace(la.LA_OP_CAUSAL_BWD_POLY, B, H, N, D, M, 1, dev)
    fwd = lambda: la.la_causal_fwd_poly(qd, kd, vd, out, den, wf, B, H, N, D, M, 1)
    bwd = lambda: la.la_causal_bwd_poly(qd, kd, vd, out, den, gd, dq, dk, dv, wb, B, H, N, D, M, 1)
    for _ in range(3):
        fwd()
        bwd()
    (mf, mb), ms = step_and_calls([fwd, bwd], 100, flush, torch, dev)
    fb, bb = causal_bytes(B, H, N, D, M, 2)
    gbs = (fb + bb) / (ms / 1e3) / 1e9
    res["causal_poly_bf16"] = {
        "value": round(B * N / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "fwd_ms": round(mf, 5), "bwd_ms": round(mb, 5), "B": B, "H": H, "N": N, "D": D, "M": M,
        "features": D * (D + 1) // 2,
        "launches": la.la_kernel_launches(la.LA_OP_CAUSAL_FWD_POLY, B, H, N, D, M, 1)
        + la.la_kernel_launches(la.LA_OP_CAUSAL_BWD_POLY, B, H, N, D, M, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": fb + bb,
                     "bytes_per_token_head": (fb + bb) // (B * H * N)},
        "timing": "CUDA events, L2 flushed before each step (100 steps)"}
    if with_cpu:
        import oracle
        cores = _cores(oracle)
        q1, k1, v1, g1 = (t[:1] for t in (q, k, v, g))  # one batch entry: H sequences
        t0 = time.perf_counter()
        oracle.causal_fwd_poly(q1, k1, v1, nthreads=cores)
        oracle.causal_bwd_poly(q1, k1, v1, g1, nthreads=cores)
        el = time.perf_counter() - t0
        res["causal_poly_bf16"]["cpu_baseline"] = {
            "value": round(N / el, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one batch entry (H={H} sequences of N={N}), fwd+bwd pairwise form, {el:.1f} s"}


def _noncausal(la, torch, dev, flush, peaks, with_cpu, res):
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, noncausal_inputs
    w = WORKLOADS["noncausal_speech_f32"]
    B, H, N, D, M = w.B, w.H, w.N, w.D, w.M
    lengths, q, k, v, g = noncausal_inputs(B, H, N, D, M, w.dtype, w.seed, w.len_range)
    qd, kd, vd, gd, ld = (t.to(dev) for t in (q, k, v, g, lengths))
    out = torch.empty_like(vd)
    den = torch.empty(B, H, N, device=dev)
    S = torch.empty(B, H, D, M, device=dev)
    Z = torch.empty(B, H, D, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wf = la.workspace(la.LA_OP_NONCAUSAL_FWD, B, H, N, D, M, 0, dev)
    wb = la.workspace(la.LA_OP_NONCAUSAL_BWD, B, H, N, D, M, 0, dev)
    fwd = lambda: la.la_noncausal_fwd(qd, kd, vd, ld, out, den, S, Z, wf, B, H, N, D, M, 0)
    bwd = lambda: la.la_noncausal_bwd(qd, kd, vd, ld, out, den, S, Z, gd, dq, dk, dv, wb, B, H, N,
                                      D, M, 0)
    for _ in range(3):
        fwd()
        bwd()
    (mf, mb), ms = step_and_calls([fwd, bwd], 50, flush, torch, dev)
    valid = int(lengths.sum()) * H  # valid token-heads
    # fwd: q, k, v in, out and den out; bwd: q, k, v, dout and den in (out is
    # not needed: gt . out = phi(Q) . S gt / den), dq, dk, dv out; valid rows only
    alg = valid * (4 * (2 * D + M) + 4 * M + 4) + valid * (4 * (2 * D + M) + 4 * M + 4 + 4 * (2 * D + M))
    flops = valid * 12 * D * M
    gbs = alg / (ms / 1e3) / 1e9
    res["noncausal_speech_f32"] = {
        "value": round(int(lengths.sum()) / (ms / 1e3), 1), "unit": "valid tokens/s",
        "ms_per_step": round(ms, 5), "fwd_ms": round(mf, 5), "bwd_ms": round(mb, 5),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": alg},
        "fp32_tflops": round(flops / (ms / 1e3) / 1e12, 2)}
    if with_cpu:
        res["noncausal_speech_f32"]["cpu_baseline"] = cpu_baseline_noncausal(q, k, v, g, lengths)



def _prefill(la, torch, dev, flush, peaks, with_cpu, res):
    """The causal forward from a state, leaving the state after the sequence
    (the 3072-token image workload's shape; the state carries over from call
    to call like consecutive prompt segments)."""
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs
    wc = WORKLOADS["causal_cifar_bf16"]
    B, H, N, D, M = wc.B, wc.H, wc.N, wc.D, wc.M
    q, k, v, _ = causal_inputs(B, H, N, D, M, wc.dtype, wc.seed)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    out = torch.empty_like(vd)
    den = torch.empty(B, H, N, device=dev)
    S = torch.zeros(B, H, D, M, device=dev)
    Z = torch.zeros(B, H, D, device=dev)
    wp = la.workspace(la.LA_OP_CAUSAL_PREFILL, B, H, N, D, M, 1, dev)
    pre = lambda: la.la_causal_prefill(qd, kd, vd, out, den, S, Z, wp, B, H, N, D, M, 1)
    for _ in range(3):
        pre()
    (mp,), _ = time_calls([pre], 50, flush, torch, None, dev)
    alg = B * H * N * (2 * (2 * D + M) + 2 * M + 4) + B * H * 2 * 4 * (D * M + D)
    gbs = alg / (mp / 1e3) / 1e9
    res["prefill_cifar_bf16"] = {
        "value": round(B * N / (mp / 1e3), 1), "unit": "tokens/s", "ms_per_call": round(mp, 5),
        "launches": la.la_kernel_launches(la.LA_OP_CAUSAL_PREFILL, B, H, N, D, M, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": alg}}
    if with_cpu:
        res["prefill_cifar_bf16"]["cpu_baseline"] = cpu_baseline_prefill(q, k, v, B, H, N)


def _decode(la, torch, dev, peaks, with_cpu, res):
    for Bd in (256, 2048):
        Hd, Dd, Md = 8, 64, 64
        S = torch.zeros(Bd, Hd, Dd, Md, device=dev)
        Z = torch.ones(Bd, Hd, Dd, device=dev)
        gen = torch.Generator(device="cpu").manual_seed(5)
        qd = torch.randn(Bd, Hd, Dd, generator=gen).to(dev)
        kd = torch.randn(Bd, Hd, Dd, generator=gen).to(dev)
        vd = torch.randn(Bd, Hd, Md, generator=gen).to(dev)
        y = torch.empty(Bd, Hd, Md, device=dev)
        stepf = lambda: la.la_decode_step(qd, kd, vd, S, Z, y, Bd, Hd, Dd, Md, 0)
        per = 64  # steps per CUDA graph replay
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                stepf()
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per):
                stepf()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * per)
        alg = Bd * Hd * (2 * 4 * Dd * Md + 2 * 4 * Dd + 4 * (2 * Dd) + 4 * 2 * Md)
        gbs = alg / (us / 1e6) / 1e9
        res[f"decode_f32_B{Bd}"] = {
            "us_per_step": round(us, 3), "unit": "us/step",
            "stream_tokens_per_s": round(Bd * Hd / (us / 1e6), 1),
            "state_bytes": Bd * Hd * (Dd * Md + Dd) * 4,
            "l2_resident": Bd * Hd * (Dd * Md + Dd) * 4 < 100e6,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": alg},
            "timing": "CUDA graph of 64 steps, 20 replays, state kept warm"}
        if with_cpu and Bd == 256:
            res[f"decode_f32_B{Bd}"]["cpu_baseline"] = cpu_baseline_decode(Bd, Hd, Dd, Md)


def _decode_proj(la, torch, dev, flush, peaks, with_cpu, res, name):
    """The decode step fed by its q/k/v projection (one launch: the bf16
    projection on the tensor cores, then the fp32 state update and read-out)."""
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, proj_inputs
    wp = WORKLOADS[name]
    B, H, D, M, dm = wp.B, wp.H, wp.D, wp.M, wp.d_model
    x, W, S0, Z0 = proj_inputs(B, dm, H, D, M, t=wp.N, seed=wp.seed)
    xd, Wd, Sd, Zd = (t.to(dev) for t in (x, W, S0, Z0))
    y = torch.empty(B, H, M, dtype=torch.bfloat16, device=dev)
    call = lambda: la.la_decode_step_proj(xd, Wd, Sd, Zd, y, B, H, dm, D, M, 1)
    for _ in range(3):
        call()
    (mp,), _ = time_calls([call], 50, flush, torch, None, dev)
    alg = proj_bytes(B, H, dm, D, M)
    flops = 2 * B * dm * H * (2 * D + M)
    gbs = alg / (mp / 1e3) / 1e9
    res[name] = {
        "value": round(B / (mp / 1e3), 1), "unit": "stream-steps/s", "us_per_step": round(mp * 1e3, 3),
        "B": B, "H": H, "D": D, "M": M, "d_model": dm,
        "launches": la.la_kernel_launches(la.LA_OP_DECODE_PROJ, B, H, dm, D, M, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "alg_bytes": alg,
                     "bytes": "x, W read once; S, Z read and written once; y written"},
        "projection_tflops": round(flops / (mp / 1e3) / 1e12, 2),
        "timing": "CUDA events per call, L2 flushed before each (50 calls)"}
    if with_cpu:
        res[name]["cpu_baseline"] = cpu_baseline_decode_proj(x, W, S0, Z0, H, D, M)


def proj_bytes(B, H, dm, D, M):
    """Algorithmic bytes of one projected decode step: x and W (bf16) read
    once, the fp32 state S, Z read and written once, y (bf16) written."""
    return B * dm * 2 + dm * H * (2 * D + M) * 2 + B * H * (2 * 4 * (D * M + D) + 2 * M)


# -------------------------------------------------------------- CPU oracle

def _cores(orc_mod):
    return orc_mod.default_threads() if orc_mod.openmp_enabled() else 1


def cpu_baseline(q, k, v, g, B, H, N, budget_s=12.0):
    """The fp64 oracle as it stands (recurrent form, fwd then bwd) on all host
    cores, repeated over the full workload until about `budget_s` seconds."""
    import oracle
    cores = _cores(oracle)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.causal_fwd(q, k, v, "recurrent", nthreads=cores)
        oracle.causal_bwd(q, k, v, g, "recurrent", nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 200:
            break
    # one core: the first (b, h) sequence alone, fwd then bwd; a token needs all H heads
    q1, k1, v1, g1 = (t[:1, :1] for t in (q, k, v, g))
    t1 = time.perf_counter()
    oracle.causal_fwd(q1, k1, v1, "recurrent", nthreads=1)
    oracle.causal_bwd(q1, k1, v1, g1, "recurrent", nthreads=1)
    t1 = time.perf_counter() - t1
    return {"value": round(reps * B * N / el, 1), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"full workload (B={B}, H={H}, N={N}) x {reps} repetitions, "
                      f"{el:.1f} s, fp64 recurrent form, fwd+bwd",
            "cpu_model": cpu_model(),
            "single_core": {"value": round(N / (H * t1), 1), "unit": "tokens/s",
                            "sample": f"one (b, h) sequence of N={N}, fwd+bwd, {t1:.2f} s, "
                                      f"scaled by 1/H"}}


def cpu_baseline_noncausal(q, k, v, g, lengths, budget_s=5.0):
    """The fp64 oracle's non-causal fwd then bwd on all host cores, over the
    full workload, repeated until about `budget_s` seconds (at least once)."""
    import oracle
    cores = _cores(oracle)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.noncausal_fwd(q, k, v, lengths, nthreads=cores)
        oracle.noncausal_bwd(q, k, v, g, lengths, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 20:
            break
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    return {"value": round(reps * int(lengths.sum()) / el, 1), "unit": "valid tokens/s",
            "cores": cores, "kind": "oracle",
            "sample": f"full workload (B={B}, H={H}, N={N}, lengths as the GPU line) x {reps}, "
                      f"{el:.1f} s, fp64, fwd+bwd"}


def cpu_baseline_prefill(q, k, v, B, H, N, budget_s=5.0):
    """The fp64 oracle's prefill (recurrent form from a zero state) on all host
    cores over the full workload, repeated until about `budget_s` seconds."""
    import oracle
    cores = _cores(oracle)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.causal_prefill(q, k, v, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 20:
            break
    return {"value": round(reps * B * N / el, 1), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"full workload (B={B}, H={H}, N={N}) x {reps}, {el:.1f} s, fp64, recurrent form"}


def cpu_baseline_decode(B, H, D, M, steps=64, budget_s=5.0):
    """The fp64 oracle's decode steps for all B x H streams on all host cores,
    `steps` steps per call (synthetic normal q, k, v), until about `budget_s`
    seconds; reported as stream-steps per second like the GPU line."""
    import numpy as np
    import oracle
    cores = _cores(oracle)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((steps, B, H, D))
    k = rng.standard_normal((steps, B, H, D))
    v = rng.standard_normal((steps, B, H, M))
    S = np.zeros((B, H, D, M))
    Z = np.ones((B, H, D))
    t0 = time.perf_counter()
    reps = 0
    while True:
        _, S, Z = oracle.decode(q, k, v, S, Z, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 200:
            break
    return {"value": round(reps * steps * B * H / el, 1), "unit": "stream-steps/s",
            "cores": cores, "kind": "oracle",
            "sample": f"B={B} x H={H} streams, {reps} x {steps} steps, {el:.1f} s, fp64"}


def cpu_baseline_decode_proj(x, W, S, Z, H, D, M, budget_s=4.0):
    """The fp64 oracle's projected decode step (numpy x @ W, then the RNN
    step) on all host cores, over the first n streams of the same inputs, n
    doubled until one call takes about a second (or all streams are in),
    repeated until about `budget_s` seconds; stream-steps per second."""
    import oracle
    cores = _cores(oracle)
    B = x.shape[0]
    n = min(B, 64)
    while True:
        t0 = time.perf_counter()
        oracle.decode_proj(x[:n], W, H, D, M, S[:n], Z[:n], nthreads=cores)
        one = time.perf_counter() - t0
        if one >= 1.0 or n >= B:
            break
        n = min(B, 2 * n)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.decode_proj(x[:n], W, H, D, M, S[:n], Z[:n], nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 100:
            break
    return {"value": round(reps * n / el, 1), "unit": "stream-steps/s", "cores": cores,
            "kind": "oracle",
            "sample": f"first {n} of {B} streams (H={H}, D={D}, M={M}, d_model={x.shape[1]}) x {reps}, "
                      f"{el:.1f} s, fp64 numpy projection + C step"}


def run_reference(args, dist):
    """The CPU oracle as the reference arm: rank 0 times K steps, each a
    bounded sample of the workload (whole heads of the N=3072 sequences)."""
    if dist.rank != 0:
        return None
    import oracle
    from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs
    w = WORKLOADS[WORKLOAD]
    B, H, N, D, M = w.B, w.H, w.N, w.D, w.M
    q, k, v, g = causal_inputs(B, H, N, D, M, w.dtype, w.seed)
    cores = _cores(oracle)
    # calibrate: one head
    t0 = time.perf_counter()
    oracle.causal_fwd(q[:1, :1], k[:1, :1], v[:1, :1], "recurrent", nthreads=1)
    oracle.causal_bwd(q[:1, :1], k[:1, :1], v[:1, :1], g[:1, :1], "recurrent", nthreads=1)
    per_head_1core = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)  # whole run within ~2.5 minutes
    heads = int(max(1, min(B * H, budget * cores / max(per_head_1core, 1e-6))))
    qs, ks, vs, gs = (t.reshape(1, B * H, N, -1)[:, :heads].contiguous() for t in (q, k, v, g))
    step = lambda: (oracle.causal_fwd(qs, ks, vs, "recurrent", nthreads=cores),
                    oracle.causal_bwd(qs, ks, vs, gs, "recurrent", nthreads=cores))
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = statistics.fmean(times) * 1e3
    tokens = heads * N / H  # a sample of whole heads counts as that fraction of the batch
    value = tokens / (ms / 1e3)
    sample = f"{heads} of {B * H} heads x N={N} per step (fp64 recurrent form, fwd+bwd)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "D": D, "M": M},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_secondary_only(only=None):
    """The secondary measurements alone (or the subset `only`), on cuda:0."""
    import torch

    import kernelized_causal_attention_gb300 as la

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    la.lib()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    return {"secondary": secondary(la, torch, dev, lambda: flush_buf.zero_(), measured_peaks(),
                                   with_cpu=False, only=only)}


def sweep_points(la, torch, dev, flush, peaks, Ns, steps, total=1 << 16):
    """Causal attention and its gradients (la_causal_fwd + la_causal_bwd) at
    each N in Ns with the batch inversely proportional to N (B * N = total),
    H = 8, D = M = 64, bf16 inputs: time and peak allocated device memory per
    sample, the shape of the pages' memory/computation benchmark (§4.1,
    Fig. 1).  Peak memory is torch's allocator high-water mark over the
    inputs, outputs, gradients and workspaces (the library allocates nothing
    itself); time is the mean of `steps` L2-flushed fwd+bwd pairs on CUDA
    events."""
    from kernelized_causal_attention_gb300.workloads import causal_inputs
    H, D, M = 8, 64, 64
    points = []
    for N in Ns:
        B = max(1, total // N)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        q, k, v, g = (t.to(dev) for t in causal_inputs(B, H, N, D, M, "bf16", 900 + N.bit_length()))
        out = torch.empty_like(v)
        den = torch.empty(B, H, N, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wf = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, 1, dev)
        wb = la.workspace(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, 1, dev)
        fwd = lambda: la.la_causal_fwd(q, k, v, out, den, wf, B, H, N, D, M, 1)
        bwd = lambda: la.la_causal_bwd(q, k, v, out, den, g, dq, dk, dv, wb, B, H, N, D, M, 1)
        for _ in range(3):
            fwd()
            bwd()
        (mf, mb), ms = step_and_calls([fwd, bwd], steps, flush, torch, dev)
        peak = torch.cuda.max_memory_allocated(dev) - base
        alg = sum(causal_bytes(B, H, N, D, M, 2))
        gbs = alg / (ms / 1e3) / 1e9
        points.append({"N": N, "B": B, "ms_fwd_bwd": round(ms, 5), "fwd_ms": round(mf, 5),
                       "bwd_ms": round(mb, 5), "ms_per_sample": round(ms / B, 6),
                       "peak_bytes": int(peak), "peak_bytes_per_sample": int(peak // B),
                       "tokens_per_s": round(B * N / (ms / 1e3), 1),
                       "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)})
        del q, k, v, g, out, den, dq, dk, dv, wf, wb
    return points


def run_sweep(steps=20):
    """The full sweep N = 2^9 .. 2^16 (B * N = 2^16) on cuda:0."""
    import torch

    import kernelized_causal_attention_gb300 as la

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    la.lib()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    points = sweep_points(la, torch, dev, lambda: flush_buf.zero_(), measured_peaks(),
                          [1 << e for e in range(9, 17)], steps)
    la.check_device_status()
    return {"sweep": "causal fwd+bwd, N = 2^9 .. 2^16, B * N = 2^16, H = 8, D = M = 64, bf16",
            "data": "synthetic", "l2": "flushed before every timed pair", "points": points}


def main():
    args = parse()
    dist = Dist()
    if args.secondary_only:
        if dist.rank == 0:
            print(json.dumps(run_secondary_only(None if args.only is None else set(args.only.split(",")))), flush=True)
        return
    if args.sweep:
        if dist.rank == 0:
            print(json.dumps(run_sweep()), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, dist)
    else:
        res = run_ours(args, dist)
    if res is not None and dist.rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
