#!/usr/bin/env python
"""Benchmark of the forward transposed convolution on GB300.

One JSON line on rank 0.  A step is one ct_conv_transpose_nd call (every
kernel of the chosen route: weight reorder, layout pass, phase GEMM or
gather, bias epilogue) over the workload's synthetic inputs, resident in HBM.
Between timed steps a 512 MiB buffer is written to flush the 129 MB L2.

metric  : ConvTranspose TFLOP/s (valid multiply-adds x 2 / time); the HBM
          GB/s (algorithmic bytes x + w + bias + y / time) and the roofline
          fraction of the dominant kernel are reported beside it.
e2e     : the same metric through ct_conv_transpose_nd_host with pinned host
          buffers (host-to-device copies of x, w, bias and the device-to-host
          copy of y inside the timed region).
backward : each gradient (dx, dw, db) of every workload timed on its own
          through ct_conv_transpose_backward_nd (skip with --no-backward).
--impl reference : the fp64 CPU oracle timed on the host cores on a bounded
          sample of the same workload (the only other place this script runs
          the oracle is the cpu_baseline leg).
Several GPUs (torchrun): independent replicas, one per rank, no collective on
the data path; value = all ranks' work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from transposed_convolution_convtranspose1_gb300 import synth  # noqa: E402

METRIC = "ConvTranspose TFLOP/s and HBM GB/s per config, as fraction of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FMA pipe: 152 SMs x 128 lanes x 2 flop x 2070 MHz maximum SM clock
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2070e6 / 1e12
# nominal dense TF32 / BF16 tensor rates (1.1 and 2.25 PFLOP/s per GPU)
TF32_PER_BF16 = 1.1 / 2.25
FLUSH_BYTES = 512 << 20


# --------------------------------------------------------------------------
# algorithmic work
# --------------------------------------------------------------------------

def _out_extent(I, k, s, pl, ph, d, op):
    return (I - 1) * s - pl - ph + d * (k - 1) + op + 1


def valid_macs(p: synth.Problem) -> int:
    """Multiply-adds whose product lands inside the output (separable per axis)."""
    per_axis = 1
    for a in range(p.nd):
        O = _out_extent(p.spatial[a], p.k[a], p.stride[a], p.pad_lo[a], p.pad_hi[a],
                        p.dilation[a], p.output_padding[a])
        n = 0
        for t in range(p.k[a]):
            for i in range(p.spatial[a]):
                o = i * p.stride[a] - p.pad_lo[a] + t * p.dilation[a]
                n += 0 <= o < O
        per_axis *= n
    return p.B * p.C_out * (p.C_in // p.groups) * per_axis


def out_shape(p):
    return tuple(_out_extent(p.spatial[a], p.k[a], p.stride[a], p.pad_lo[a], p.pad_hi[a],
                             p.dilation[a], p.output_padding[a]) for a in range(p.nd))


def alg_bytes(p: synth.Problem) -> int:
    eb = torch.tensor([], dtype=p.torch_dtype).element_size()
    x = p.B * p.C_in * math.prod(p.spatial)
    w = p.C_in * (p.C_out // p.groups) * math.prod(p.k)
    b = p.C_out if p.bias else 0
    y = p.B * p.C_out * math.prod(out_shape(p))
    return (x + w + b + y) * eb


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Each dominant kernel (named by the library's ct_conv_transpose_kernel): the
# bound that applies to it and the source file its DRAM traffic figure
# depends on.
KERNEL_INFO = {
    "gather_kernel": ("alu", "ct_gather.cu"),
    "grouped_warp_kernel": ("hbm", "ct_grouped_warp.cu"),
    "grouped_tma_kernel": ("hbm", "ct_grouped_tma.cu"),
    "grouped_staged_kernel": ("hbm", "ct_grouped.cu"),
    "grouped_kernel": ("hbm", "ct_grouped.cu"),
    "simt_phase_gemm": ("alu", "ct_simt.cu"),
    "tc_phase_gemm": ("tensor", "ct_tc.cu"),
    "tc32_phase_gemm": ("tensor", "ct_tc32.cu"),
    "bias_fill_kernel": ("hbm", "ct_gather.cu"),
}


# How each route computes (the JSON line's dtype is the operand/output type).
ARITHMETIC = {
    "tc32_gemm": "f32 operands split into TF32 hi + lo; hi*hi + hi*lo + lo*hi on tcgen05 "
                 "kind::tf32, fp32 accumulation",
    "simt_gemm": "f32 FMA",
    "tc_gemm": "bf16/f16 operands, fp32 accumulation on tcgen05 kind::f16",
}


def _src_sha(fname):
    path = os.path.join(ROOT, "transposed_convolution_convtranspose1_gb300", "csrc", fname)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel, workload):
    """(DRAM bytes of the dominant kernel, whole-call traffic) from the
    committed capture (profiles/traffic.json), while the source of every
    kernel of the call still matches; (None, None) otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    e = d.get("workloads", {}).get(workload)
    if not e or any(_src_sha(src) != h for src, h in e.get("sources", {}).items()):
        return None, None
    k = e["kernels"].get(kernel)
    kernel_bytes = None if k is None else k["dram_read"] + k["dram_write"]
    c = e["call"]
    call = {"dram_read": c["dram_read"], "sm_write": c["sm_write"], "traffic": c["traffic"],
            "vs_algorithmic": round(c["traffic"] / e["algorithmic_bytes"], 3)}
    return kernel_bytes, call


def dominant_kernel(p):
    """The kernel the library runs for p's main work (ct_conv_transpose_kernel)."""
    import transposed_convolution_convtranspose1_gb300 as ct
    return ct.ct_conv_transpose_kernel(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                       p.pad_hi, p.dilation, p.output_padding, p.groups,
                                       ct.dtype_code(p.torch_dtype))


def roofline(route_name, p, main_ms, peaks, timed_alone):
    kernel = dominant_kernel(p)
    bound, _ = KERNEL_INFO.get(kernel, ("hbm", "ct_gather.cu"))
    if route_name in ("gather", "simt_gemm") and p.dtype != "f32":
        bound = "alu"
    flops = 2.0 * valid_macs(p)
    nbytes = alg_bytes(p)
    if bound == "tensor":
        peak = peaks["bf16_tflops"] if timed_alone else peaks.get("bf16_tflops_sustained",
                                                                  peaks["bf16_tflops"])
        basis = "bf16 tensor peak"
        if route_name == "tc32_gemm":
            # three TF32 products per fp32 product: the fp32 work rate the
            # TF32 pipe can sustain is a third of its peak
            peak = peak * TF32_PER_BF16 / 3.0
            basis = "bf16 tensor peak x nominal tf32/bf16 (1.1/2.25) / 3 TF32 products per fp32 product"
        achieved = flops / (main_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    elif bound == "alu":
        peak = FP32_ALU_PEAK_TFLOPS
        basis = "nominal fp32 FMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz"
        achieved = flops / (main_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        peak = peaks["hbm_gbs"]
        basis = "HBM copy bandwidth"
        achieved = nbytes / (main_ms * 1e-3) / 1e9
        unit = "GB/s"
    kernel_bytes, call = traffic_for(kernel, p.name)
    return {"bound": bound, "kernel": kernel, "achieved": round(achieved, 3),
            "peak": round(peak, 3), "unit": unit, "frac": round(achieved / peak, 4),
            "peak_basis": basis, "traffic": kernel_bytes, "call_traffic": call,
            "algorithmic_bytes": nbytes, "algorithmic_flop": flops}


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

def _smi_device_id(local):
    """nvidia-smi's id for this process's GPU (UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[local].strip()
    return str(local)


class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="ct_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for r in csv.reader(f):
                    if len(r) >= 10:
                        rows.append([c.strip() for c in r])
            os.unlink(self.path)
        return self._summary(rows)

    def _summary(self, rows):
        def ts(r):
            # nvidia-smi writes local time as "YYYY/MM/DD HH:MM:SS.mmm"
            try:
                whole, _, frac = r[0].partition(".")
                t = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S"))
                return t + (float("0." + frac) if frac else 0.0)
            except Exception:
                return None
        # samples whose timestamps fall inside the timed region; when the region is
        # shorter than the sampling period and none does, the nearest ones
        # within 0.25 s of it, said so in "window"
        inside = [r for r in rows if ts(r) is not None and self.t0 is not None
                  and self.t0 <= ts(r) <= (self.t1 or 1e18)]
        window = "timed region"
        use = inside
        if not use and self.t0 is not None:
            use = [r for r in rows if ts(r) is not None
                   and self.t0 - 0.25 <= ts(r) <= (self.t1 or 1e18) + 0.25]
            window = "within 0.25 s of the timed region (none fell inside it)"
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0, "samples_in_timed_region": 0}
        sm = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside), "window": window}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def _workload_problem(spec):
    try:
        return synth.workload(int(spec))
    except ValueError:
        return synth.workload(spec)


class Runner:
    """Device buffers and one-step closure for a workload."""

    def __init__(self, p, dev):
        import transposed_convolution_convtranspose1_gb300 as ct
        self.ct = ct
        self.p = p
        x, w, b = synth.make_inputs(p)
        self.x, self.w = x.to(dev), w.to(dev)
        self.b = None if b is None else b.to(dev)
        self.y = torch.empty((p.B, p.C_out) + out_shape(p), dtype=p.torch_dtype, device=dev)
        nws = ct.ct_conv_transpose_workspace_bytes(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
        self.ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
        self.route = ct.ct_conv_transpose_route(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
        self.host = None

    def step(self, m0=None, m1=None):
        p = self.p
        return self.ct.ct_conv_transpose_nd_profiled(
            self.x, self.w, self.b, self.y, self.ws, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, main_start=m0, main_stop=m1)

    def host_step(self):
        p = self.p
        if self.host is None:
            self.host = (self.x.cpu().pin_memory(), self.w.cpu().pin_memory(),
                         None if self.b is None else self.b.cpu().pin_memory(),
                         torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory())
        hx, hw, hb, hy = self.host
        self.ct.ct_conv_transpose_nd_host(hx, hw, hb, hy, p.stride, p.pad_lo, p.pad_hi,
                                          p.dilation, p.output_padding, p.groups)

    def h2d_d2h_bytes(self):
        eb = self.y.element_size()
        h2d = (self.x.numel() + self.w.numel() + (0 if self.b is None else self.b.numel())) * eb
        return h2d, self.y.numel() * eb


def _events(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:  # create the handles so the library can record them
        e.record()
    return evs


def time_steps(r: Runner, K, flush):
    """K steps; per step: flush L2, then events around the call and its main kernel."""
    e0, e1, m0, m1 = _events(K), _events(K), _events(K), _events(K)
    torch.cuda.synchronize()
    launches = 0
    for i in range(K):
        if flush is not None:
            flush.add_(1)
        e0[i].record()
        n, _ = r.step(m0[i], m1[i])
        e1[i].record()
        launches += n
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
    main_ms = [a.elapsed_time(b) for a, b in zip(m0, m1)]
    return step_ms, main_ms, launches


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the initialised process group:
    the slowest rank sets every time the job reports."""
    t = torch.tensor(values, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def run_ours(args):
    import transposed_convolution_convtranspose1_gb300 as ct
    from transposed_convolution_convtranspose1_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        _build.build_library()
    if world > 1:
        torch.distributed.barrier()
    ct.lib()

    p = _workload_problem(args.config)
    peaks, peak_src = load_peaks()
    r = Runner(p, dev)
    flush = None if args.no_flush else torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32,
                                                   device=dev)
    W = max(args.warmup, 3)
    for _ in range(W):
        r.step()
    torch.cuda.synchronize()
    # steps: exactly --steps K when given; otherwise enough for >= 2 s of timed work
    if args.steps > 0:
        K = args.steps
    else:
        t = time_steps(r, 5, flush)[0]
        K = int(min(2000, max(20, math.ceil(2000.0 / max(statistics.median(t), 1e-3)))))

    clocks = ClockSampler(_smi_device_id(local))
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark_begin()
    wall0 = time.perf_counter()
    step_ms, main_ms, launches = time_steps(r, K, flush)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    clocks.mark_end()
    clk = clocks.stop()

    # one statistic everywhere: the median step (and dominant-kernel) time
    ms = statistics.median(step_ms)
    main = statistics.median(main_ms)
    if world > 1:
        ms, main = max_over_ranks([ms, main], dev)

    flops = 2.0 * valid_macs(p)
    nbytes = alg_bytes(p)
    value = world * flops / (ms * 1e-3) / 1e12
    route_name = ct.ROUTE_NAMES.get(r.route, str(r.route))

    # e2e through the host-buffer entry point
    for _ in range(2):
        r.host_step()
    Ke = max(3, min(K, 20))
    t0 = time.perf_counter()
    for _ in range(Ke):
        r.host_step()
    e2e_s = (time.perf_counter() - t0) / Ke
    if world > 1:
        (e2e_s,) = max_over_ranks([e2e_s], dev)
    h2d, d2h = r.h2d_d2h_bytes()

    rl = roofline(route_name, p, main, peaks, timed_alone=True)
    rl["peak_source"] = "nominal" if rl["bound"] == "alu" else peak_src
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": p.dtype, "data": "synthetic",
        "config": {"workload": p.name, "B": p.B, "C_in": p.C_in, "C_out": p.C_out,
                   "spatial": list(p.spatial), "k": list(p.k), "stride": list(p.stride),
                   "pad_lo": list(p.pad_lo), "pad_hi": list(p.pad_hi),
                   "dilation": list(p.dilation), "output_padding": list(p.output_padding),
                   "groups": p.groups, "bias": p.bias, "route": route_name,
                   "arithmetic": ARITHMETIC.get(route_name, p.dtype),
                   "l2": "flushed between timed steps (512 MiB write)" if flush is not None
                   else "not flushed", "parallelism": f"replicas x{world}"},
        "hbm_gbs": round(world * nbytes / (ms * 1e-3) / 1e9, 2),
        "main_kernel_ms": round(main, 5),
        "roofline": rl,
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 4), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4), "api": "ct_conv_transpose_nd_host"},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": round(wall1 - wall0, 4),
    }

    # the bulky objects first and per_config last, compact, so that the tail a
    # log keeps of this one line still holds every workload's figures
    if not args.no_backward and world == 1:
        line["backward"] = backward_per_config(dev, flush, peaks)
        if rank == 0 and not args.no_cpu_baseline:
            line["backward"]["cpu_baseline"] = backward_cpu_baseline(p, min(args.cpu_seconds, 10.0))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, args.cpu_seconds)
    if not args.no_per_config and world == 1:
        line["per_config"] = per_config(args, dev, peaks, flush, skip=p.name)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def per_config(args, dev, peaks, flush, skip):
    """Every workload, 20 L2-flushed steps each, medians: call time (ms),
    dominant-kernel time (kernel_ms) and that kernel's roofline fraction."""
    import transposed_convolution_convtranspose1_gb300 as ct
    out = {}
    for p in synth.WORKLOADS:
        r = Runner(p, dev)
        for _ in range(3):
            r.step()
        torch.cuda.synchronize()
        K = 20
        step_ms, main_ms, _ = time_steps(r, K, flush)
        ms, main = statistics.median(step_ms), statistics.median(main_ms)
        route_name = ct.ROUTE_NAMES.get(r.route, str(r.route))
        flops = 2.0 * valid_macs(p)
        rl = roofline(route_name, p, main, peaks, timed_alone=True)
        out[p.name] = {
            "route": route_name, "kernel": rl["kernel"], "ms": round(ms, 5),
            "kernel_ms": round(main, 5), "tflops": round(flops / (ms * 1e-3) / 1e12, 3),
            "bound": rl["bound"], "achieved": rl["achieved"], "unit": rl["unit"],
            "frac": rl["frac"], "traffic": rl["traffic"],
            "call_traffic_ratio": rl["call_traffic"]["vs_algorithmic"] if rl["call_traffic"] else None}
        del r
        torch.cuda.empty_cache()
    return out


def backward_per_config(dev, flush, peaks):
    """Each gradient of every workload timed on its own (events around a call
    that requests only it, L2 flushed before each), as [median ms, fraction]:
    dx and dw against the fp32 FMA peak on the CUDA-core kernels, against the
    measured bf16 tensor peak where the gradient runs on the tensor cores
    (third element "t"; work = the forward's 2 x valid MACs each), db against
    HBM bandwidth (dy read once)."""
    import transposed_convolution_convtranspose1_gb300 as ct
    out = {"format": "[ms, fraction of peak]: dx, dw of the fp32 FMA peak (of the bf16 tensor peak "
                     "when marked t: tcgen05 kernel; of the 3xTF32 peak when marked t32), db of HBM"}
    for p in synth.WORKLOADS:
        x, w, _ = synth.make_inputs(p)
        x, w = x.to(dev), w.to(dev)
        O = out_shape(p)
        g = torch.Generator().manual_seed(4242)
        dy = torch.randn((p.B, p.C_out) + O, generator=g).to(p.torch_dtype).to(dev)
        dx, dw = torch.empty_like(x), torch.empty_like(w)
        db = torch.empty((p.C_out,), dtype=dy.dtype, device=dev)
        nws = ct.ct_conv_transpose_backward_workspace_bytes(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
        flops = 2.0 * valid_macs(p)
        kern = dict(zip(("dx", "dw"), ct.ct_conv_transpose_backward_kernels(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))))
        res = {}
        for name, args in (("dx", (dx, None, None)), ("dw", (None, dw, None)),
                           ("db", (None, None, db))):
            def call():
                ct.ct_conv_transpose_backward_nd(x, w, dy, *args, ws, p.stride, p.pad_lo,
                                                 p.pad_hi, p.dilation, p.output_padding, p.groups)
            for _ in range(3):
                call()
            K = 10
            e0, e1 = _events(K), _events(K)
            torch.cuda.synchronize()
            for i in range(K):
                if flush is not None:
                    flush.add_(1)
                e0[i].record()
                call()
                e1[i].record()
            torch.cuda.synchronize()
            ms = statistics.median([a.elapsed_time(b) for a, b in zip(e0, e1)])
            if name == "db":
                nbytes = dy.numel() * dy.element_size() + p.C_out * dy.element_size()
                ach = nbytes / (ms * 1e-3) / 1e9
                res[name] = [round(ms, 5), round(ach / peaks["hbm_gbs"], 4)]
            elif kern[name] == "tc32_phase_gemm":
                # fp32 on TF32 tensor cores, three products each: the 3xTF32 peak
                ach = flops / (ms * 1e-3) / 1e12
                res[name] = [round(ms, 5), round(ach / (peaks["bf16_tflops"] * TF32_PER_BF16 / 3), 4), "t32"]
            elif kern[name] in ("tc_phase_gemm", "tc_dw_gemm"):
                ach = flops / (ms * 1e-3) / 1e12
                res[name] = [round(ms, 5), round(ach / peaks["bf16_tflops"], 4), "t"]
            else:
                ach = flops / (ms * 1e-3) / 1e12
                res[name] = [round(ms, 5), round(ach / FP32_ALU_PEAK_TFLOPS, 4)]
        out[p.name] = res
        del x, w, dy, dx, dw, db, ws
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------

def _oracle_sample(p, target_s):
    """A sub-batch of the workload sized for about target_s seconds of oracle time."""
    import oracle
    x, w, b = synth.make_inputs(p)
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.conv_transpose(x[:1], w, b, **p.attrs(), threads=threads)
    t1 = time.perf_counter() - t0
    nb = int(max(1, min(p.B, math.floor(target_s / max(t1, 1e-6)))))
    return x, w, b, nb, threads


def cpu_baseline(p, target_s):
    """The oracle on the host cores: a sub-batch sized for about target_s
    seconds, repeated (up to 20 times) until about target_s have elapsed."""
    import oracle
    x, w, b, nb, threads = _oracle_sample(p, target_s)
    times = []
    while not times or (sum(times) < target_s and len(times) < 20):
        t0 = time.perf_counter()
        oracle.conv_transpose(x[:nb], w, b, **p.attrs(), threads=threads)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    flops = 2.0 * valid_macs(p.replace(B=nb))
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(sum(times), 3), "runs": len(times),
            "sample": f"batch elements 0..{nb - 1} of {p.B} of {p.name} (fp64 scatter-add, "
                      f"{threads} threads), {len(times)} runs"}


def backward_cpu_baseline(p, target_s):
    """The backward oracle (dx and dw, fp64) on the host cores on one batch
    element of the workload, repeated until about target_s have elapsed."""
    import oracle
    x, w, _ = synth.make_inputs(p.replace(B=1))
    O = out_shape(p)
    g = torch.Generator().manual_seed(4242)
    dy = torch.randn((1, p.C_out) + O, generator=g).to(p.torch_dtype)
    threads = os.cpu_count() or 1
    times = []
    while not times or (sum(times) < target_s and len(times) < 10):
        t0 = time.perf_counter()
        oracle.conv_transpose_backward(x, w, dy, **p.attrs(), threads=threads, need=("dx", "dw"))
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    flops = 2.0 * 2.0 * valid_macs(p.replace(B=1))  # dx and dw, each the forward's work
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(sum(times), 3), "runs": len(times),
            "sample": f"dx and dw of batch element 0 of {p.B} of {p.name} (fp64 adjoint "
                      f"scatter, {threads} threads), {len(times)} runs"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    p = _workload_problem(args.config)
    steps = args.steps if args.steps > 0 else 3
    per_step = max(1.0, min(20.0, 60.0 / max(steps + args.warmup, 1)))
    x, w, b, nb, threads = _oracle_sample(p, per_step)
    for _ in range(min(args.warmup, 1)):
        oracle.conv_transpose(x[:nb], w, b, **p.attrs(), threads=threads)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.conv_transpose(x[:nb], w, b, **p.attrs(), threads=threads)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    flops = 2.0 * valid_macs(p.replace(B=nb))
    value = flops / dt / 1e12
    sample = f"batch elements 0..{nb - 1} of {p.B} of {p.name} per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": p.name, "route": "oracle (CPU fp64 scatter-add)"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: enough for about 2 s of timed work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="1", help="workload index 0-4 or name (default 1)")
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the per-workload gradient timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
