#!/usr/bin/env python3
"""Benchmark of the forward 2-D convolution library on one or more GPUs.

Workload (one "step"): the 4-layer MSCRED signature-matrix encoder in fp32
NCHW on a batch of 256 time steps of 3x30x30 signature matrices
(3->32 3x3 s1p1, 32->64 3x3 s2p1, 64->128 2x2 s2p1, 128->256 2x2 s2p0, each
with bias, each layer fed by the previous one).  Metric: conv2d forward
TFLOPS = sum over layers of 2*N*K*P*Q*C*R*S / time, plus the roofline
fraction of the dominant kernel and the extra workspace (always 0 bytes).

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream; a step is one replay of a CUDA graph holding the 4 C-ABI
launches, with the L2 flush (a 256 MiB write) and the two timing events
captured inside the same graph, so the events bracket only the 4 kernels:
neither host-side validation nor the graph launch latency sits inside them.
Barrier + synchronize on both sides of the timed region; the slowest rank's
time is reported.  With --gpus N > 1 (torchrun) every rank runs an
independent replica of the workload (the layer needs no exchange), so the
total work grows with N ("weak" scaling).

Beside the step the JSON line carries: every encoder layer and every
fp16/bf16 layer timed alone (--layer-iters replays, 10 warm-ups, L2 flushed
before each, median / mean / min), the single signature-matrix convolution
and the 1x1 kernel-size-sweep layer also as a CUDA graph of 100 back-to-back
launches (the per-call floor), the eager step and the host time of one C-ABI
call, the end-to-end step (`e2e`: pinned-host x copied in, the 4 layers, y
copied out to pinned host, all inside the timed region; one CUDA graph per
step like `value`, and also as eager calls and as a pipelined stream of
batches), the step with the fp32
tensor-core (3xTF32) path off, the fp32 FFMA / TF32 / BF16 MMA peaks measured
by the library's probe kernels (the fp32 roofline denominators), and the
nvidia-smi clocks sampled across every GPU leg.

The cpu_baseline leg times the fp64 oracle on the host cores (all cores, and
one core for the single convolution and layer 1) and compares the bench's own
GPU outputs (encoder layers, fp16/bf16 layers, single convolution) with it at
random, border and per-tile sample points.

--impl reference times the fp64 CPU oracle on the same workload (a bounded
sample of it) on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "conv2d fwd TFLOPS (2·NKPQCRS/t) and % of GB300 roofline; extra workspace bytes"
WORKLOAD = "mscred_encoder_4layer_f32_nchw_n256_c3_30x30"
L2_FLUSH_BYTES = 256 << 20
SMS = 152
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


def fp32_alu_peak_tflops(peaks=None):
    """FFMA peak: the probe kernel's measurement of this run when there is one,
    else SMs x 128 lanes x 2 x the maximum SM clock."""
    if peaks and peaks.get("ffma_tflops_probe"):
        return peaks["ffma_tflops_probe"]
    return SMS * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12


# DRAM bytes (read + write) per launch of a layer's kernel, from one ncu
# capture of the kernel with the plan given here (profiles/ holds the summary
# and command); a plan that differs gets null.
DRAM_TRAFFIC = {
    # profiles/tf32x3_conv_kernel_mscred_encoder_l2.md
    ("mscred_enc_l2_n256_c32_30x30_k64_3x3s2p1",
     "tensor_core tcgen05 3xtf32 BM=128 BN=64 BK=32 stages=2 producers=512 groups=2 resident-w grid=152 "
     "smem=218496"): 29629184,
}

# nominal dense TF32 / BF16 tensor rates of GB300 (1.1 and 2.25 PFLOP/s), used
# only when the probe measurement is missing
TF32_PER_BF16 = 1.1 / 2.25


def fp32_3xtf32_peak_tflops(peaks):
    """fp32 convolution on tensor cores as three TF32 products per multiply-add:
    the measured TF32 MMA rate / 3."""
    if peaks.get("tf32_mma_tflops_probe"):
        return peaks["tf32_mma_tflops_probe"] / 3.0
    return peaks["bf16_tflops"] * TF32_PER_BF16 / 3.0


def layer_peak(plan, peaks):
    """(bound, peak TFLOP/s, source) for the kernel a plan string names."""
    if plan.startswith("tensor_core tcgen05 3xtf32"):
        if peaks.get("tf32_mma_tflops_probe"):
            return ("tensor", fp32_3xtf32_peak_tflops(peaks),
                    f"measured TF32 MMA rate {peaks['tf32_mma_tflops_probe']:.1f} TFLOP/s "
                    "(conv2d_peak_probe, this run) / 3 TF32 products per fp32 multiply-add")
        return ("tensor", fp32_3xtf32_peak_tflops(peaks),
                f"measured bf16 {peaks['bf16_tflops']} TFLOP/s x nominal TF32/BF16 (1.1/2.25) / 3")
    if peaks.get("ffma_tflops_probe"):
        return ("alu", fp32_alu_peak_tflops(peaks),
                "measured FFMA rate (conv2d_peak_probe, this run)")
    return ("alu", fp32_alu_peak_tflops(), "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz")


def measure_probe_peaks(reps=5):
    """TFLOP/s of the library's FFMA, TF32-MMA and BF16-MMA probe kernels
    (best of `reps` timings of three back-to-back launches of a few ms each,
    CUDA events)."""
    from cnn_convolution_gb300 import conv2d
    out = {}
    for kind, iters in (("ffma", 4000), ("tf32_mma", 12000), ("bf16_mma", 12000)):
        conv2d.peak_probe(kind, max(1, iters // 8))
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(reps):
            # three launches between the events: the host time of a call
            # overlaps the previous launch instead of sitting in the interval
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(1_000_000)
            e0.record()
            fl = sum(conv2d.peak_probe(kind, iters) for _ in range(3))
            e1.record()
            e1.synchronize()
            best = max(best, fl / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        out[f"{kind}_tflops_probe"] = round(best, 2)
    if conv2d.get_device_status() != 0:
        raise RuntimeError("a probe kernel reported a barrier timeout")
    return out


# ------------------------------------------------------------------ distributed

def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 50 ms from start()
    to stop(); summary() covers a time window (default: all samples)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.samples = []          # (perf_counter time, line)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def wait_first(self, timeout=5.0):
        t0 = time.perf_counter()
        while self.proc is not None and not self.samples and time.perf_counter() - t0 < timeout:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)
            self.proc = None

    def summary(self, t0=None, t1=None):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in list(self.samples):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(power), "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload

def encoder_setup(device):
    from cnn_convolution_gb300 import conv2d, workloads as wl
    x = wl.mscred_encoder_input(256)
    params = wl.mscred_encoder_params()
    descs, ws, bs, outs = [], [], [], []
    for spec, (w, b) in zip(wl.MSCRED_ENCODER, params):
        d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S,
                              spec.stride, spec.pad, spec.dil, torch.float32, "NCHW")
        descs.append(d)
        ws.append(w.to(device))
        bs.append(b.to(device))
        outs.append(torch.empty(d.y_shape(), dtype=torch.float32, device=device))
    flops = []
    for spec, d in zip(wl.MSCRED_ENCODER, descs):
        P, Q = d.output_dims()
        flops.append(2.0 * spec.N * spec.K * P * Q * spec.C * spec.R * spec.S)
    return wl.MSCRED_ENCODER, x, descs, ws, bs, outs, flops


def layer_bytes(spec, P, Q):
    elt = {"f32": 4, "f16": 2, "bf16": 2}[spec.dtype]
    n = (spec.N * spec.C * spec.H * spec.W + spec.K * spec.C * spec.R * spec.S +
         (spec.K if spec.bias else 0) + spec.N * spec.K * P * Q)
    return n * elt


def run_encoder(descs, x_dev, ws, bs, outs, events=None):
    cur = x_dev
    for i, d in enumerate(descs):
        if events is not None:
            events[i].record()
        d.forward(cur, ws[i], bs[i], y=outs[i])
        cur = outs[i]
    if events is not None:
        events[len(descs)].record()
    return cur


def e2e_pipelined(descs, x_host, ws, bs, outs, steps, warmup):
    """ms per batch of a stream of encoder batches through the C ABI, with the
    copies overlapped with compute: batch i's input is copied in on one stream
    (pinned host -> device) while batch i-1 computes, and its output copied out
    on another while batch i+1 computes.  Two input buffers, two last-layer
    outputs and two pinned output buffers alternate; events order every reuse.
    Timed from the first copy-in to the last copy-out of `steps` batches."""
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    x_pin = [x_host.pin_memory(), x_host.clone().pin_memory()]
    x_buf = [torch.empty(x_host.shape, dtype=x_host.dtype, device="cuda") for _ in range(2)]
    y_last = [outs[-1], torch.empty_like(outs[-1])]
    y_pin = [torch.empty(outs[-1].shape, dtype=outs[-1].dtype).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_l1 = [torch.cuda.Event() for _ in range(2)]     # layer 1 has read x_buf[slot]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def batch(i):
        k = i % 2
        if i >= 2:
            s_in.wait_event(ev_l1[k])
        with torch.cuda.stream(s_in):
            x_buf[k].copy_(x_pin[k], non_blocking=True)
            ev_in[k].record(s_in)
        comp.wait_event(ev_in[k])
        if i >= 2:
            comp.wait_event(ev_out[k])                  # y_last[k] has been copied out
        cur = x_buf[k]
        for j, d in enumerate(descs):
            y = y_last[k] if j == len(descs) - 1 else outs[j]
            d.forward(cur, ws[j], bs[j], y=y)
            if j == 0:
                ev_l1[k].record(comp)
            cur = y
        ev_comp[k].record(comp)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            y_pin[k].copy_(y_last[k], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(warmup):
        batch(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        batch(i)
    e1.record(s_out)
    e1.synchronize()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def capture(fn):
    """Capture fn's launches (on a side stream, as torch requires) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def timing_event():
    """A timing event that can be recorded inside a captured CUDA graph."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:   # older torch without graph-external events
        return None


class TimedGraph:
    """One CUDA graph holding [L2 flush, event, fn's launches, event].

    The events are recorded inside the graph, so a replay's elapsed time covers
    only fn's kernels: neither the graph launch latency nor the flush.  Where
    graph-external events are unavailable, the events bracket the replay from
    outside (launch latency included)."""

    def __init__(self, fn, flush):
        self.e0, self.e1 = timing_event(), timing_event()
        self.inside = self.e0 is not None
        if not self.inside:
            self.e0 = torch.cuda.Event(enable_timing=True)
            self.e1 = torch.cuda.Event(enable_timing=True)
        self.flush = flush
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g):
            if self.inside:
                flush.zero_()
                self.e0.record()
            fn()
            if self.inside:
                self.e1.record()

    def replay_ms(self):
        if self.inside:
            self.g.replay()
        else:
            self.flush.zero_()
            self.e0.record()
            self.g.replay()
            self.e1.record()
        self.e1.synchronize()
        return self.e0.elapsed_time(self.e1)


def time_graph(tg, iters, warm=10):
    """Replay a TimedGraph `warm` times, then `iters` times; (median, mean, min) ms."""
    for _ in range(warm):
        tg.replay_ms()
    ts = [tg.replay_ms() for _ in range(iters)]
    return statistics.median(ts), statistics.mean(ts), min(ts)


def graph_floor_us(fn, n=100, reps=5):
    """Per-call time of `fn` in a CUDA graph of n back-to-back calls (no L2
    flush between them): the launch-and-tail floor of a small layer."""
    g = capture(lambda: [fn() for _ in range(n)])
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / n)
    return best


def single_conv_leg(device, flush, iters, peaks):
    """The single signature-matrix convolution (1x3x30x30 -> 32, 3x3, fp32):
    one launch after an L2 flush, and the per-call floor of 100 launches."""
    from cnn_convolution_gb300 import conv2d, workloads as wl
    spec = wl.MSCRED_SINGLE
    x, w, b = wl.mscred_single_inputs()
    d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride,
                          spec.pad, spec.dil, torch.float32, "NCHW")
    xd, wd, bd = x.to(device), w.to(device), b.to(device)
    y = torch.empty(d.y_shape(), dtype=torch.float32, device=device)
    for _ in range(3):
        d.forward(xd, wd, bd, y=y)
    torch.cuda.synchronize()
    med, mean, mn = time_graph(TimedGraph(lambda: d.forward(xd, wd, bd, y=y), flush), iters)
    floor = graph_floor_us(lambda: d.forward(xd, wd, bd, y=y))
    P, Q = d.output_dims()
    fl = 2.0 * spec.N * spec.K * P * Q * spec.C * spec.R * spec.S
    d.forward(xd, wd, bd, y=y)
    torch.cuda.synchronize()
    res = {"layer": spec.name, "plan": d.plan(), "us_median": round(med * 1e3, 3),
           "us_min": round(mn * 1e3, 3), "tflops": round(fl / (med * 1e-3) / 1e12, 4),
           "graph_100_per_call_us": round(floor, 3),
           "graph_100_tflops": round(fl / (floor * 1e-6) / 1e12, 4), "bound": "latency",
           "workspace_bytes": d.workspace_bytes(), "iters": iters}
    idx = np.stack([a.reshape(-1) for a in np.indices((spec.N, spec.K, P, Q))], axis=1)
    return res, (spec, x, w, b, idx, wl.gather_points(y, idx, "NCHW").cpu())


def bench_main(args):
    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    from cnn_convolution_gb300 import conv2d, workloads as wl
    conv2d.load()
    peaks, peak_src = load_peaks()
    peaks = dict(peaks)

    clk = ClockSampler(device.index).start()
    clk.wait_first()
    t_gpu0 = time.perf_counter()
    peaks.update(measure_probe_peaks())

    specs, x_host, descs, ws, bs, outs, flops = encoder_setup(device)
    x_dev = x_host.to(device)
    step_flops = sum(flops)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    n_layers = len(descs)

    # Eager warm-up (plans, tensor maps), then one CUDA graph for the whole
    # 4-layer step and one per layer (per-layer times for the roofline).
    for _ in range(args.warmup):
        run_encoder(descs, x_dev, ws, bs, outs)
    torch.cuda.synchronize()
    step_graph = TimedGraph(lambda: run_encoder(descs, x_dev, ws, bs, outs), flush)
    layer_graphs = []
    for i in range(n_layers):
        src = x_dev if i == 0 else outs[i - 1]
        layer_graphs.append(TimedGraph(
            lambda i=i, src=src: descs[i].forward(src, ws[i], bs[i], y=outs[i]), flush))
    torch.cuda.synchronize()

    step_ms = []
    for _ in range(args.warmup):
        step_graph.replay_ms()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        step_ms.append(step_graph.replay_ms())
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    barrier(world)
    local_ms = statistics.mean(step_ms)
    ms = max_over_ranks(local_ms, world)
    value = step_flops * world / (ms * 1e-3) / 1e12

    # per-layer launches, each alone after an L2 flush (not part of the step time)
    layer_t = [time_graph(layer_graphs[i], args.layer_iters) for i in range(n_layers)]

    # eager step (every call through the C ABI from Python, host overhead included)
    eager = []
    for _ in range(max(10, args.steps // 4)):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run_encoder(descs, x_dev, ws, bs, outs)
        e1.record()
        e1.synchronize()
        eager.append(e0.elapsed_time(e1))
    # host time of one C-ABI call (validation, plan lookup, launch), GPU kept busy meanwhile
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)
    t0 = time.perf_counter()
    n_calls = 200
    for _ in range(n_calls // n_layers):
        run_encoder(descs, x_dev, ws, bs, outs)
    host_us = (time.perf_counter() - t0) / (n_calls // n_layers * n_layers) * 1e6
    torch.cuda.synchronize()
    # the same through the raw C ABI (argument marshalling done once): the
    # library's own host time per call (validation, plan lookup, launch)
    import ctypes
    lib = conv2d.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    raw = []
    for i, d in enumerate(descs):
        src = x_dev if i == 0 else outs[i - 1]
        raw.append((d.handle, src.data_ptr(), ws[i].data_ptr(), bs[i].data_ptr(), outs[i].data_ptr()))
    torch.cuda._sleep(50_000_000)
    t0 = time.perf_counter()
    for _ in range(n_calls // n_layers):
        for h, xp, wp, bp, yp in raw:
            lib.conv2d_forward_desc(h, xp, wp, bp, yp, st)
    host_us_c = (time.perf_counter() - t0) / (n_calls // n_layers * n_layers) * 1e6
    torch.cuda.synchronize()

    # per-layer roofline; the dominant kernel is the layer with the largest time
    layers = []
    for i, (spec, d) in enumerate(zip(specs, descs)):
        P, Q = d.output_dims()
        med, mean, mn = layer_t[i]
        tf = flops[i] / (mean * 1e-3) / 1e12
        gbs = layer_bytes(spec, P, Q) / (mean * 1e-3) / 1e9
        bound, cpeak, _ = layer_peak(d.plan(), peaks)
        layers.append({"layer": spec.name, "plan": d.plan(), "ms": round(mean, 5),
                       "ms_median": round(med, 5), "ms_min": round(mn, 5),
                       "tflops": round(tf, 3), "bound": bound, "peak": round(cpeak, 2),
                       "compute_frac": round(tf / cpeak, 4),
                       "alu_frac": round(tf / fp32_alu_peak_tflops(peaks), 4),
                       "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                       "iters": args.layer_iters})
    dom = max(range(n_layers), key=lambda i: layer_t[i][1])
    dom_t = layer_t[dom][1]
    achieved = flops[dom] / (dom_t * 1e-3) / 1e12
    dom_bound, dom_peak, dom_src = layer_peak(descs[dom].plan(), peaks)
    traffic = DRAM_TRAFFIC.get((specs[dom].name, descs[dom].plan()))
    roofline = {"kernel": specs[dom].name, "plan": descs[dom].plan(), "bound": dom_bound,
                "achieved": round(achieved, 3), "peak": round(dom_peak, 2), "unit": "TFLOP/s",
                "frac": round(achieved / dom_peak, 4), "traffic": traffic, "peak_source": dom_src,
                "duration_us": round(dom_t * 1e3, 3),
                "algorithmic_flops_per_launch": flops[dom]}

    # end to end through the C ABI: pinned host x -> device, 4 layers, y -> pinned host
    x_pin = x_host.pin_memory()
    y_pin = torch.empty(outs[-1].shape, dtype=torch.float32).pin_memory()
    x_buf = torch.empty_like(x_dev)
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        x_buf.copy_(x_pin, non_blocking=True)
        run_encoder(descs, x_buf, ws, bs, outs)
        y_pin.copy_(outs[-1], non_blocking=True)
        e1.record()
        e1.synchronize()
        if it >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    eager_t = max_over_ranks(statistics.mean(e2e_ms), world)
    # the same step launched like `value`: one CUDA graph holding the copy-in,
    # the 4 C-ABI calls and the copy-out, events inside it, L2 flushed first
    def e2e_body():
        x_buf.copy_(x_pin, non_blocking=True)
        run_encoder(descs, x_buf, ws, bs, outs)
        y_pin.copy_(outs[-1], non_blocking=True)
    e2e_graph = TimedGraph(e2e_body, flush)
    for _ in range(args.warmup):
        e2e_graph.replay_ms()
    e2e_t = max_over_ranks(statistics.mean([e2e_graph.replay_ms() for _ in range(args.steps)]), world)
    pipe_t = max_over_ranks(e2e_pipelined(descs, x_host, ws, bs, outs, args.steps, args.warmup), world)

    # the two copies alone (CUDA events, median of 20): what the host link costs
    def copy_us(fn):
        ts = []
        for it in range(25):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            if it >= 5:
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)
    h2d_us = copy_us(lambda: x_buf.copy_(x_pin, non_blocking=True))
    d2h_us = copy_us(lambda: y_pin.copy_(outs[-1], non_blocking=True))
    e2e = {"value": round(step_flops * world / (e2e_t * 1e-3) / 1e12, 4), "unit": "TFLOPS",
           "ms_per_step": round(e2e_t, 5),
           "h2d_bytes_per_step": x_pin.numel() * 4, "d2h_bytes_per_step": y_pin.numel() * 4,
           "launch": "one CUDA graph per step (as for `value`): pinned-host x copied in, the 4 "
                     "C-ABI calls, y copied out to pinned host, timing events inside the graph; "
                     "one step at a time, L2 flushed before each",
           "copies_alone": {"h2d_us": round(h2d_us, 2), "d2h_us": round(d2h_us, 2),
                            "h2d_gbs": round(x_pin.numel() * 4 / (h2d_us * 1e3), 1),
                            "d2h_gbs": round(y_pin.numel() * 4 / (d2h_us * 1e3), 1)},
           "eager": {"value": round(step_flops * world / (eager_t * 1e-3) / 1e12, 4),
                     "unit": "TFLOPS", "ms_per_step": round(eager_t, 5),
                     "note": "the same step as eager C-ABI calls from Python (host overhead "
                             "included), events around it"},
           "pipelined": {"value": round(step_flops * world / (pipe_t * 1e-3) / 1e12, 4),
                         "unit": "TFLOPS", "ms_per_step": round(pipe_t, 5),
                         "note": "a stream of batches: batch i+1's H2D copy and batch i-1's D2H "
                                 "copy run on their own streams while batch i computes "
                                 "(double-buffered; every batch's copies inside the timed region; "
                                 "no L2 flush between batches)"}}

    # the step's outputs, for the oracle check of the cpu_baseline leg: each
    # layer's sampled outputs and the input that layer received
    run_encoder(descs, x_dev, ws, bs, outs)
    torch.cuda.synchronize()
    enc_check = []
    for i, (spec, d) in enumerate(zip(specs, descs)):
        P, Q = d.output_dims()
        idx = wl.check_points(spec, P, Q, seed=i)
        src = x_host if i == 0 else outs[i - 1].cpu()
        enc_check.append((spec, src, ws[i].cpu(), bs[i].cpu(), idx,
                          wl.gather_points(outs[i], idx, "NCHW").cpu()))

    # the same step with the fp32 tensor-core (3xTF32) path switched off:
    # every layer on CUDA-core FFMA kernels (direct / implicit GEMM)
    with conv2d.overrides(fp32_tc=0):
        for _ in range(2):
            run_encoder(descs, x_dev, ws, bs, outs)
        torch.cuda.synchronize()
        cc_graph = TimedGraph(lambda: run_encoder(descs, x_dev, ws, bs, outs), flush)
        cc_plans = [d.plan() for d in descs]
        cc_ms = [cc_graph.replay_ms() for _ in range(max(10, args.steps // 4))]
    cc_t = max_over_ranks(statistics.mean(cc_ms), world)
    fp32_cuda_core_only = {"value": round(step_flops * world / (cc_t * 1e-3) / 1e12, 4),
                           "unit": "TFLOPS", "ms_per_step": round(cc_t, 5), "plans": cc_plans}

    # signature matrices on the GPU: the kernel alone (its roofline is the
    # HBM traffic of series slice + output), and the encoder end to end from
    # the raw signals (pinned host series -> signature kernel -> 4 layers ->
    # pinned host y), which moves 38 KB to the device instead of 2.8 MB
    sig = signature_stage(device, flush, descs, ws, bs, outs, peaks, args, world)

    single, single_check = single_conv_leg(device, flush, args.layer_iters, peaks) \
        if rank == 0 else (None, None)
    cells = convlstm_cells(device, flush, peaks, iters=args.layer_iters) if rank == 0 else []
    decoder = decoder_layers(device, flush, peaks, iters=args.layer_iters) if rank == 0 else []

    extra, tc_check = [], []
    if not args.no_tensor_core and rank == 0:
        extra, tc_check = tensor_core_layers(device, peaks, flush, iters=args.layer_iters,
                                             keep_check=True)
    torch.cuda.synchronize()
    t_gpu1 = time.perf_counter()
    clk.stop()
    clocks = clk.summary(t_gpu0, t_gpu1)
    clocks["window"] = "every GPU leg of this run (probe peaks through the fp16/bf16 layers)"
    step_clk = clk.summary(t_wall0, t_wall1)
    clocks["timed_region_samples"] = step_clk["samples"]
    clocks["timed_region_sm_mhz"] = step_clk["sm_mhz"]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x_host, [(w.cpu(), b.cpu()) for w, b in zip(ws, bs)], specs, flops,
                           checks=enc_check + tc_check + ([single_check] if single_check else []))

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 4), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random-walk signature matrices; Kaiming-uniform weights)",
            "config": {"workload": WORKLOAD, "global_batch": 256 * world, "layers": 4,
                       "layout": "NCHW", "l2": "flushed before every timed step (256 MiB write)",
                       "launch": "CUDA graph of the 4 C-ABI calls; timing events inside the graph",
                       "parallelism": "replicas" if world > 1 else "single_gpu"},
            "workspace_bytes": 0,
            "roofline": roofline,
            "layers": layers,
            "eager_ms_per_step": round(statistics.mean(eager), 5),
            "host_us_per_call": round(host_us, 2),
            "host_us_per_call_c_abi": round(host_us_c, 2),
            "e2e": e2e,
            "fp32_cuda_core_only": fp32_cuda_core_only,
            "single_signature_conv": single,
            "signature_matrices": sig,
            "convlstm_cells": cells,
            "decoder_deconv_layers": decoder,
            "gpu_launches": n_layers * args.steps,
            "clocks": clocks,
            "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"],
                      "bf16_tflops": peaks["bf16_tflops"],
                      "ffma_tflops_probe": peaks.get("ffma_tflops_probe"),
                      "tf32_mma_tflops_probe": peaks.get("tf32_mma_tflops_probe"),
                      "bf16_mma_tflops_probe": peaks.get("bf16_mma_tflops_probe"),
                      "fp32_3xtf32_tflops": round(fp32_3xtf32_peak_tflops(peaks), 2),
                      "probe": "conv2d_peak_probe kernels, best of 5 launches, CUDA events"},
            "wall_s_timed_region": round(t_wall1 - t_wall0, 4),
            "tensor_core_layers": extra,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def signature_stage(device, flush, descs, ws, bs, outs, peaks, args, world):
    from cnn_convolution_gb300 import conv2d, workloads as wl
    n = 256
    windows = list(wl.MSCRED_WINDOWS)
    series_host = wl.mscred_encoder_series(n)
    series = series_host.to(device)
    x_sig = torch.empty((n, len(windows), 30, 30), dtype=torch.float32, device=device)
    for _ in range(3):
        conv2d.signature_matrices(series, windows, 60, n, out=x_sig)
    torch.cuda.synchronize()
    tg = TimedGraph(lambda: conv2d.signature_matrices(series, windows, 60, n, out=x_sig), flush)
    ts = [tg.replay_ms() for _ in range(max(10, args.steps // 4))]
    t = statistics.median(ts)
    # algorithmic bytes: the series samples the end times read, once, and the output
    read = series_host.shape[0] * (60 + n - 1) * 4
    written = x_sig.numel() * 4
    gbs = (read + written) / (t * 1e-3) / 1e9
    # end to end from the raw signals, through the C ABI
    s_pin = series_host.pin_memory()
    y_pin = torch.empty(outs[-1].shape, dtype=torch.float32).pin_memory()
    s_buf = torch.empty_like(series)
    e2e = []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        s_buf.copy_(s_pin, non_blocking=True)
        conv2d.signature_matrices(s_buf, windows, 60, n, out=x_sig)
        run_encoder(descs, x_sig, ws, bs, outs)
        y_pin.copy_(outs[-1], non_blocking=True)
        e1.record()
        e1.synchronize()
        if it >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    e2e_t = max_over_ranks(statistics.mean(e2e), world)
    enc_flops = 0.0
    for d in descs:
        N, C, H, W, K, R, S, st, pad, dil = d.sizes
        P, Q = d.output_dims()
        enc_flops += 2.0 * N * K * P * Q * C * R * S
    return {"us": round(t * 1e3, 3), "shape": [n, len(windows), 30, 30], "windows": windows,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "bound": "hbm", "algorithmic_bytes": read + written,
            "e2e_from_series": {"value": round(enc_flops * world / (e2e_t * 1e-3) / 1e12, 4),
                                "unit": "TFLOPS", "ms_per_step": round(e2e_t, 5),
                                "h2d_bytes_per_step": s_pin.numel() * 4,
                                "d2h_bytes_per_step": y_pin.numel() * 4,
                                "note": "signature kernel + 4 layers, eager C-ABI calls"}}


def convlstm_cells(device, flush, peaks, iters, n=64):
    """One fused ConvLSTM cell step per MSCRED scale (Cx = Ch = the encoder
    layer's channels, 3x3 gates, batch n), timed alone after an L2 flush.
    FLOPs = those of the gate convolution (2*N*4Ch*H*W*(Cx+Ch)*9)."""
    from cnn_convolution_gb300 import conv2d, workloads as wl
    out = []
    peak = fp32_3xtf32_peak_tflops(peaks)
    for ch, hw in ((32, 30), (64, 15), (128, 8), (256, 4)):
        spec = wl.ConvSpec(f"convlstm_cell_n{n}_c{ch}_{hw}x{hw}_3x3", n, 2 * ch, hw, hw, 4 * ch, 3, 3, 1, 1)
        xh, w, b = wl.random_inputs(spec, seed=ch)
        xh, w, b = xh.to(device), w.to(device), b.to(device)
        c0 = torch.zeros(n, ch, hw, hw, device=device)
        c1, h1 = torch.empty_like(c0), torch.empty_like(c0)
        for _ in range(3):
            conv2d.convlstm_cell(xh, w, b, c0, 1, c_next=c1, h_next=h1)
        torch.cuda.synchronize()
        tg = TimedGraph(lambda: conv2d.convlstm_cell(xh, w, b, c0, 1, c_next=c1, h_next=h1), flush)
        ts = [tg.replay_ms() for _ in range(iters)]
        t = statistics.median(ts)
        fl = 2.0 * n * 4 * ch * hw * hw * 2 * ch * 9
        tf = fl / (t * 1e-3) / 1e12
        out.append({"cell": spec.name, "us": round(t * 1e3, 2), "tflops": round(tf, 2),
                    "bound": "tensor", "peak": round(peak, 1), "frac": round(tf / peak, 4)})
    return out


def decoder_layers(device, flush, peaks, iters, n=256):
    """The MSCRED decoder's transposed convolutions (fp32 NCHW, batch n), each
    timed alone after an L2 flush.  FLOPs count the products that land inside
    the output: 2 * N * K * C * (valid (p, r) pairs) * (valid (q, s) pairs)."""
    from cnn_convolution_gb300 import conv2d
    shapes = [("deconv4_256to128_4to8_2x2s2", 256, 4, 128, 2, 2, 0, 0),
              ("deconv3_256to64_8to15_3x3s2", 256, 8, 64, 3, 2, 1, 0),
              ("deconv2_128to32_15to30_3x3s2", 128, 15, 32, 3, 2, 1, 1),
              ("deconv1_64to3_30to30_3x3s1", 64, 30, 3, 3, 1, 1, 0)]
    out = []
    g = torch.Generator().manual_seed(7)
    for name, K, P, C, R, st, pad, op in shapes:
        x = torch.randn((n, K, P, P), generator=g).to(device)
        w = (torch.randn((K, C, R, R), generator=g) / math.sqrt(K * R * R)).to(device)
        b = torch.zeros(C).to(device)
        H, W = conv2d.deconv_output_dims(P, P, R, R, st, pad, 1, op)
        y = torch.empty((n, C, H, W), device=device)
        for _ in range(3):
            conv2d.deconv_forward(x, w, b, st, pad, 1, op, y=y)
        torch.cuda.synchronize()
        tg = TimedGraph(lambda: conv2d.deconv_forward(x, w, b, st, pad, 1, op, y=y), flush)
        t = statistics.median([tg.replay_ms() for _ in range(iters)])
        valid = sum(1 for p in range(P) for r in range(R) if 0 <= p * st - pad + r < H)
        fl = 2.0 * n * K * C * valid * valid
        by = 4.0 * (x.numel() + w.numel() + C + y.numel())
        tf = fl / (t * 1e-3) / 1e12
        gbs = by / (t * 1e-3) / 1e9
        if C > 8:   # the library's rule: tensor cores unless the layer has <= 8 output channels
            path, bound, peak = ("3xTF32 tensor cores, one launch per output residue class", "tensor",
                                 fp32_3xtf32_peak_tflops(peaks))
        else:
            path = ("FFMA, one image per CTA, 4 pixels x %d channels per thread" % (4 if C <= 4 else 8)
                    if st == 1 else "gather kernel, FFMA, %d-channel block" % (4 if C <= 4 else 8))
            bound, peak = "alu", fp32_alu_peak_tflops(peaks)
        out.append({"layer": name, "us": round(t * 1e3, 2), "tflops": round(tf, 2), "path": path,
                    "bound": bound, "frac": round(tf / peak, 4), "hbm_gbs": round(gbs, 1)})
    return out


def time_layer(d, x, w, b, y, flush, iters, warm=10):
    """(median, mean, min) kernel time of one layer, L2 flushed before each launch."""
    for _ in range(3):
        d.forward(x, w, b, y=y)
    torch.cuda.synchronize()
    return time_graph(TimedGraph(lambda: d.forward(x, w, b, y=y), flush), iters, warm)


def tensor_core_layers(device, peaks, flush, iters=50, names=None, keep_check=False):
    """Time each fp16/bf16 NHWC layer alone (L2 flushed before each launch).

    With `names`, time those layers instead (any named layer, fp32 included).
    With keep_check, also return each layer's sampled outputs (and inputs) for
    the oracle check of the cpu_baseline leg."""
    from cnn_convolution_gb300 import conv2d, workloads as wl
    res, checks = [], []
    tc_peak = peaks["bf16_tflops"]
    specs = [wl.ALL_LAYERS[n] for n in names] if names else wl.TENSOR_CORE_WORKLOADS
    for spec in specs:
        x, w, b = wl.workload_inputs(spec)
        d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S,
                              spec.stride, spec.pad, spec.dil, spec.torch_dtype, spec.layout)
        xd, wd = x.to(device), w.to(device)
        bd = None if b is None else b.to(device)
        y = torch.empty(d.y_shape(), dtype=spec.torch_dtype, device=device)
        med, mean, mn = time_layer(d, xd, wd, bd, y, flush, iters)
        P, Q = d.output_dims()
        fl = 2.0 * spec.N * spec.K * P * Q * spec.C * spec.R * spec.S
        by = layer_bytes(spec, P, Q)
        tf = fl / (med * 1e-3) / 1e12
        gbs = by / (med * 1e-3) / 1e9
        unit, cpeak = ("tensor", tc_peak) if spec.dtype != "f32" else layer_peak(d.plan(), peaks)[:2]
        roof_t = max(fl / (cpeak * 1e12), by / (peaks["hbm_gbs"] * 1e9)) * 1e3
        bound = unit if fl / (cpeak * 1e12) >= by / (peaks["hbm_gbs"] * 1e9) else "hbm"
        row = {"layer": spec.name, "plan": d.plan(), "ms_median": round(med, 5),
               "ms_mean": round(mean, 5), "ms_min": round(mn, 5), "tflops": round(tf, 2),
               "hbm_gbs": round(gbs, 1), "bound": bound, "roofline_frac": round(roof_t / med, 4),
               "compute_frac": round(tf / cpeak, 4), "workspace_bytes": d.workspace_bytes(),
               "iters": iters}
        if spec.R == 1 and spec.S == 1 and names is None:
            # launch-bound at 3.8 us of HBM time: also the per-call floor of
            # 100 back-to-back launches (x stays in L2 between them)
            row["graph_100_per_call_us"] = round(
                graph_floor_us(lambda: d.forward(xd, wd, bd, y=y)), 3)
        res.append(row)
        if keep_check:
            d.forward(xd, wd, bd, y=y)
            idx = wl.check_points(spec, P, Q, seed=11)
            checks.append((spec, x, w, b, idx, wl.gather_points(y, idx, spec.layout).cpu()))
        del xd, wd, bd, y
    return (res, checks) if keep_check else res


# ------------------------------------------------------------------ CPU oracle

def cpu_baseline(x, params, specs, flops, budget_s=10.0, checks=()):
    """The fp64 oracle on the host cores: whole encoder steps, repeated within a
    budget, on all cores; one-core times of the single signature-matrix
    convolution and of encoder layer 1 (a slice of its batch); and the oracle
    at the sample points of the bench's own GPU outputs (error ratios)."""
    import oracle
    from cnn_convolution_gb300 import workloads as wl
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    reps = 0
    while True:
        cur = x
        for spec, (w, b) in zip(specs, params):
            y, _ = oracle.conv2d(cur, w, b, spec.stride, spec.pad, spec.dil, threads=threads)
            cur = y
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 20:
            break
    per = el / reps
    # one core: the single convolution, and layer 1 on 32 of its 256 images
    sx, sw, sb = wl.mscred_single_inputs()
    t0 = time.perf_counter()
    oracle.conv2d(sx, sw, sb, 1, 1, 1, threads=1)
    single_1t = time.perf_counter() - t0
    l1 = specs[0]
    w1, b1 = params[0]
    t0 = time.perf_counter()
    oracle.conv2d(x[:32], w1, b1, l1.stride, l1.pad, l1.dil, threads=1)
    l1_1t = (time.perf_counter() - t0) * 256 / 32
    oracle.conv2d(sx, sw, sb, 1, 1, 1, threads=threads)   # restore the thread count
    single_fl = 2.0 * 32 * 30 * 30 * 27
    res = {"value": round(sum(flops) / per / 1e12, 6), "unit": "TFLOPS", "cores": threads,
           "kind": "oracle",
           "sample": f"{reps} full encoder steps (batch 256, 4 layers), fp64 direct loop, "
                     f"{per:.3f} s per step",
           "one_core": {"single_signature_conv_s": round(single_1t, 6),
                        "single_signature_conv_tflops": round(single_fl / single_1t / 1e12, 6),
                        "encoder_layer1_s": round(l1_1t, 4),
                        "encoder_layer1_tflops": round(flops[0] / l1_1t / 1e12, 6),
                        "sample": "layer 1 timed on 32 of 256 images, scaled to 256"}}
    if checks:
        errs, ok, points = {}, True, 0
        for spec, cx, cw, cb, idx, got in checks:
            y_ref, den = oracle.conv2d_points(cx, cw, cb, idx, spec.stride, spec.pad, spec.dil,
                                              layout=spec.layout, threads=threads)
            err = oracle.error_ratio(got, y_ref, den)
            tol = 1e-6 if spec.dtype == "f32" else 4e-3
            errs[spec.name] = float(f"{err:.3e}")
            ok = ok and err <= tol
            points += len(idx)
        res["output_check"] = {"error_ratio": errs, "within_tolerance": ok, "points": points,
                               "tolerance": {"f32": 1e-6, "f16": 4e-3, "bf16": 4e-3},
                               "points_are": "random, borders of the first and last image, first "
                                             "and last row of every 128-row M tile and of every "
                                             "output row, one channel per 32-channel group"}
    return res


def reference_main(args):
    """--impl reference: the oracle on the host cores, rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from cnn_convolution_gb300 import workloads as wl
    oracle.build()
    x = wl.mscred_encoder_input(256)
    params = wl.mscred_encoder_params()
    specs = wl.MSCRED_ENCODER
    flops = []
    h = 30
    for spec in specs:
        P = oracle.out_extent(spec.H, spec.R, spec.stride, spec.pad, spec.dil)
        Q = oracle.out_extent(spec.W, spec.S, spec.stride, spec.pad, spec.dil)
        flops.append(2.0 * spec.N * spec.K * P * Q * spec.C * spec.R * spec.S)
    # each step: a bounded sample of the batch (n_img images) through the 4 layers
    n_img = int(os.environ.get("CONV2D_REF_IMAGES", "256"))
    xs = x[:n_img]
    sample_flops = sum(flops) * n_img / 256
    for _ in range(args.warmup):
        pass   # the oracle has nothing to warm up
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cur = xs
        for spec, (w, b) in zip(specs, params):
            cur, _ = oracle.conv2d(cur, w, b, spec.stride, spec.pad, spec.dil)
        times.append(time.perf_counter() - t0)
    per = statistics.mean(times)
    value = sample_flops / per / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "global_batch": 256, "layers": 4, "layout": "NCHW",
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS",
                            "cores": oracle.max_threads(), "kind": "oracle",
                            "sample": f"{n_img} of 256 images per step through all 4 layers"},
           "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-tensor-core", action="store_true", help="skip the fp16/bf16 layers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layer-iters", type=int, default=50,
                    help="timed replays per single-layer measurement (median reported)")
    ap.add_argument("--layer", default=None,
                    help="time one named layer (or signature_matrices, or mscred_encoder_step) only, for profiling, "
                         "and print its line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and args.layer is None:
        ap.error("--warmup must be at least 3")
    if args.layer_iters < 1:
        ap.error("--layer-iters must be positive")
    if args.impl == "reference":
        return reference_main(args)
    if args.layer:
        from cnn_convolution_gb300 import conv2d, workloads as wl
        conv2d.load()
        peaks, _ = load_peaks()
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        if args.layer == "mscred_encoder_step":
            # the 4-layer encoder step alone, eager, L2 flushed before each step
            specs, x_host, descs, ws, bs, outs, flops = encoder_setup(torch.device("cuda", 0))
            x_dev = x_host.cuda()
            ts = []
            for _ in range(args.steps):
                flush.zero_()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                run_encoder(descs, x_dev, ws, bs, outs)
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            print(json.dumps({"mscred_encoder_step": {"us_mean": round(statistics.mean(ts) * 1e3, 3),
                                                      "plans": [d.plan() for d in descs], "steps": args.steps}}))
            return 0
        if args.layer == "signature_matrices":
            # the encoder batch's signature matrices alone (256 end times, 30 signals)
            n, windows = 256, list(wl.MSCRED_WINDOWS)
            series = wl.mscred_encoder_series(n).cuda()
            x_sig = torch.empty((n, len(windows), 30, 30), dtype=torch.float32, device="cuda")
            tg = TimedGraph(lambda: conv2d.signature_matrices(series, windows, 60, n, out=x_sig), flush)
            med, mean, mn = time_graph(tg, args.steps)
            print(json.dumps({"signature_matrices": {"us_median": round(med * 1e3, 3),
                                                     "us_min": round(mn * 1e3, 3), "iters": args.steps}}))
            return 0
        res = tensor_core_layers(torch.device("cuda", 0), peaks, flush, iters=args.steps,
                                 names={args.layer})
        print(json.dumps({"layers": res}))
        return 0
    return bench_main(args)


if __name__ == "__main__":
    sys.exit(main())
