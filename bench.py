"""Benchmark of the implicit-GEMM convolution path on GB300.

One step = one pass of the whole hot path over one batch: for each of the
five ResNet-50-shaped layers (batch 128, bf16, NHWC) the forward pass with
bias + ReLU, the data gradient and the weight gradient, all through the C ABI
with inputs already resident in HBM.  The metric is the one the workloads are
quoted on: convolution TFLOP/s (2*N*P*Q*K*C*R*S per pass), and the fraction of
the dense bf16 tensor peak.

Prints one JSON line (rank 0).  The step is timed as a CUDA graph of its
calls between two events, with nothing between the kernels.  Keys beyond
the required ones:
  passes      per-pass TFLOP/s, from graphs of the five calls of one pass
              kind each
  layers      per-call times, from a graph with an event pair around every
              call (those event nodes add a few us per call)
  roofline    the implicit-GEMM kernel (fprop + dgrad launches, which are
              single-kernel calls) against the measured bf16 peak
  cpu_baseline the CPU oracle, timed on a bounded sample of the same workload
  e2e         the same step through the C ABI with host buffers: pinned
              host -> device copies of every input and device -> host copies
              of every output inside the timed region, pipelined over the
              layers on three streams (copies in, passes, copies out)
  rows        the other hot-path rows measured in the same run: permutes
              (GB/s), strided/dilated dgrad and wgrad layers, int8 fprop
  l2_warm     the same step replayed without the L2 flush in between
  check       seeded samples of every output the last timed step wrote,
              compared with the CPU oracle (per-element bound)
  device_status the library's device error word after every timed region
              (a kernel whose bounded wait gave up would otherwise post a
              faster time); any error ends the run with a non-zero exit code

--impl reference times the CPU oracle on bounded samples of the same
workload (there is no other implementation to run here).
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

import torch  # noqa: E402

from synthetic import (GROUPED_SWEEP, RESNET50_SWEEP, WORKLOADS, make_inputs,  # noqa: E402
                       make_inputs3d, sample_indices)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20

# DRAM bytes (read + written) per launch of the implicit-GEMM kernel: the mean
# over the 10 fprop/dgrad launches of one step, each captured alone by ncu
# (dram__bytes_read.sum + dram__bytes_write.sum, cold caches), keyed by the
# kernel source hash (SHA-256 prefix of the kernel, its launchers, its PTX
# wrappers and its parameter header).  A changed kernel source reports null
# until it is measured again.
MEASURED_TRAFFIC = {"2990eb063bae77e8": 65.03e6, "676dfad8af80c5ea": 64.11e6,
                    "cc81fa63eda9488a": 64.68e6, "53837066960d6501": 63.97e6,
                    "8c57c5a08801b7fd": 63.98e6, "abae718c2b1f3ec2": 63.97e6}


def conv_flops(pb, P, Q):
    return 2.0 * pb["N"] * P * Q * pb["K"] * pb["C"] * pb["R"] * pb["S"]


def out_hw(pb):
    def o(i, p, d, k, s):
        return (i + 2 * p - d * (k - 1) - 1) // s + 1
    return (o(pb["H"], pb["pad_h"], pb["dil_h"], pb["R"], pb["stride_h"]),
            o(pb["W"], pb["pad_w"], pb["dil_w"], pb["S"], pb["stride_w"]))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    """sha256 prefix over the implicit-GEMM kernel's sources (the kernel, its
    launchers, its PTX wrappers and the shared parameter header)."""
    h = hashlib.sha256()
    for name in ("conv_gemm_kernel.cuh", "conv_gemm.cu", "conv_gemm_s16.cu", "ptx.cuh",
                 "igconv_internal.h"):
        with open(os.path.join(ROOT, "convolution_implicit_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.gpu = str(device.index or 0)
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            if uuid:
                self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
class Layer:
    def __init__(self, name, batch=None, device="cuda"):
        import convolution_implicit_gemm_gb300 as igc
        self.igc = igc
        wl = WORKLOADS[name]
        self.name = name
        self.pb = dict(wl["problem"])
        if batch:
            self.pb["N"] = batch
        self.dtype = wl["dtype"]
        self.dw_dtype = wl.get("dw_dtype", wl["dtype"])
        self.bias = wl.get("bias", False)
        self.relu = wl.get("relu", False)
        self.groups = wl.get("groups", 1)
        self.P, self.Q = igc.conv2d_output_size(self.pb)
        self.cpu = make_inputs(self.pb, self.P, self.Q, wl["dtype"], wl["recipe"], wl["seed"],
                               bias=self.bias, dw_dtype=self.dw_dtype, groups=self.groups)
        t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
        self.td, self.tdw = t[self.dtype], t[self.dw_dtype]
        self.X = self.cpu["X"].to(device)
        self.W = self.cpu["W"].to(device)
        self.dY = self.cpu["dY"].to(device)
        self.b = self.cpu["bias"].to(device) if self.bias else None
        pb = self.pb
        self.Y = torch.empty((pb["N"], self.P, self.Q, pb["K"]), dtype=self.td, device=device)
        self.dX = torch.empty((pb["N"], pb["H"], pb["W"], pb["C"]), dtype=self.td, device=device)
        self.dW = torch.empty((pb["K"], pb["R"], pb["S"], pb["C"] // self.groups), dtype=self.tdw,
                              device=device)
        self.ws_bytes = igc.conv2d_grouped_wgrad_workspace_size(pb, self.groups, self.td,
                                                                self.tdw)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        # few input channels: fprop's pixel and filter copies; more channels:
        # the split-K partials, when the plan splits
        self.fws_bytes = igc.conv2d_fprop_workspace_size(pb, self.td)
        self.fws = (torch.empty(self.fws_bytes, dtype=torch.uint8, device=device)
                    if self.fws_bytes else None)
        # unit-stride dgrad: the split-K workspace, when the plan splits
        self.dws_bytes = (igc.conv2d_dgrad_workspace_size(pb, self.td) if self.groups == 1 else 0)
        self.dws = (torch.empty(self.dws_bytes, dtype=torch.uint8, device=device)
                    if self.dws_bytes else None)
        self.flops = conv_flops(pb, self.P, self.Q) / self.groups
        # grouped: the workspace that opens the tensor-core fprop / dgrad path
        self.gws_bytes = (igc.conv2d_grouped_fprop_workspace_size(pb, self.groups, self.td)
                          if self.groups > 1 else 0)
        self.gws = torch.empty(max(self.gws_bytes, 16), dtype=torch.uint8, device=device)

    def fprop(self):
        if self.groups > 1:
            self.igc.conv2d_grouped_fprop_ws(self.pb, self.groups, self.td, self.X, self.W,
                                             self.b, None, self.Y, 1.0, 0.0, self.relu, self.gws)
        elif self.fws is not None:
            self.igc.conv2d_fprop_ws(self.pb, self.td, self.X, self.W, self.b, None, self.Y, 1.0,
                                     0.0, self.relu, self.fws)
        else:
            self.igc.conv2d_fprop(self.pb, self.td, self.X, self.W, self.b, None, self.Y, 1.0,
                                  0.0, self.relu)

    def dgrad(self):
        if self.groups > 1:
            self.igc.conv2d_grouped_dgrad_ws(self.pb, self.groups, self.td, self.dY, self.W, None,
                                             self.dX, 1.0, 0.0, self.gws)
        elif self.dws is not None:
            self.igc.conv2d_dgrad_ws(self.pb, self.td, self.dY, self.W, None, self.dX, 1.0, 0.0,
                                     self.dws)
        else:
            self.igc.conv2d_dgrad(self.pb, self.td, self.dY, self.W, None, self.dX, 1.0, 0.0)

    def wgrad(self):
        if self.groups > 1:
            self.igc.conv2d_grouped_wgrad(self.pb, self.groups, self.td, self.tdw, self.X,
                                          self.dY, None, self.dW, 1.0, 0.0, self.ws,
                                          self.ws_bytes)
        else:
            self.igc.conv2d_wgrad(self.pb, self.td, self.tdw, self.X, self.dY, None, self.dW,
                                  1.0, 0.0, self.ws, self.ws_bytes)

    # host-side buffers for the end-to-end measurement
    def make_host(self):
        pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
        self.hX, self.hW, self.hdY = pin(self.cpu["X"]), pin(self.cpu["W"]), pin(self.cpu["dY"])
        self.hb = pin(self.cpu["bias"]) if self.bias else None
        self.hY = torch.empty(self.Y.shape, dtype=self.td).pin_memory()
        self.hdX = torch.empty(self.dX.shape, dtype=self.td).pin_memory()
        self.hdW = torch.empty(self.dW.shape, dtype=self.tdw).pin_memory()
        ins = [self.hX, self.hW, self.hdY] + ([self.hb] if self.bias else [])
        outs = [self.hY, self.hdX, self.hdW]
        self.h2d = sum(t.numel() * t.element_size() for t in ins)
        self.d2h = sum(t.numel() * t.element_size() for t in outs)

    def copy_in(self):
        for copy in self.copy_in_parts():
            copy()

    def copy_in_parts(self):
        """fprop's inputs (X, W, bias), then dY (dgrad and wgrad)."""
        def fwd():
            self.X.copy_(self.hX, non_blocking=True)
            self.W.copy_(self.hW, non_blocking=True)
            if self.bias:
                self.b.copy_(self.hb, non_blocking=True)
        return fwd, lambda: self.dY.copy_(self.hdY, non_blocking=True)

    def compute(self):
        self.fprop()
        self.dgrad()
        self.wgrad()

    def copy_out(self):
        for copy in self.copy_out_parts():
            copy()

    def copy_out_parts(self):
        """The three result copies, in pass order (Y, dX, dW)."""
        return (lambda: self.hY.copy_(self.Y, non_blocking=True),
                lambda: self.hdX.copy_(self.dX, non_blocking=True),
                lambda: self.hdW.copy_(self.dW, non_blocking=True))


class E2EPipeline:
    """One end-to-end step through the C ABI with host buffers: every layer's
    inputs copied from pinned host memory on one stream (X and W before dY,
    so fprop can start first), its three passes on a second stream once
    their own inputs have landed, and each pass's result
    copied back on a third as soon as that pass is done (Y after fprop, dX
    after dgrad, dW after wgrad).  The two copy directions run at the same
    time (the host link carries ~210 GB/s in, ~190 out, ~336 together), so
    the step's floor is its bytes over the combined rate plus the first
    layer's input copy and the last layer's output copy, which nothing
    overlaps: the layers are taken smallest input first and smallest output
    last.  The step starts and ends on `main`, so consecutive steps never
    overlap."""

    def __init__(self, layers, main):
        rest = list(layers)
        first = min(rest, key=lambda L: L.h2d)
        rest.remove(first)
        last = min(rest, key=lambda L: L.d2h) if rest else None
        if last is not None:
            rest.remove(last)
        self.layers = [first] + rest + ([last] if last is not None else [])
        self.main = main
        self.s_in, self.s_c, self.s_out = (torch.cuda.Stream() for _ in range(3))
        self.ev_in = [[torch.cuda.Event() for _ in range(2)] for _ in self.layers]
        self.ev_pass = [[torch.cuda.Event() for _ in range(3)] for _ in self.layers]

    def step(self):
        for st in (self.s_in, self.s_c, self.s_out):
            st.wait_stream(self.main)
        with torch.cuda.stream(self.s_in):
            for L, evs in zip(self.layers, self.ev_in):
                for copy, ev in zip(L.copy_in_parts(), evs):
                    copy()
                    ev.record(self.s_in)
        for L, ei, evs in zip(self.layers, self.ev_in, self.ev_pass):
            # fprop needs X and W only; dgrad and wgrad also dY
            for run, need, ev in zip((L.fprop, L.dgrad, L.wgrad), (ei[0], ei[1], ei[1]), evs):
                self.s_c.wait_event(need)
                with torch.cuda.stream(self.s_c):
                    run()
                    ev.record(self.s_c)
            for copy, ev in zip(L.copy_out_parts(), evs):
                self.s_out.wait_event(ev)
                with torch.cuda.stream(self.s_out):
                    copy()
        self.main.wait_stream(self.s_in)
        self.main.wait_stream(self.s_c)
        self.main.wait_stream(self.s_out)


def timed_launches(fn, stream):
    """Runs fn between two events on `stream`; returns the event pair."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    return a, b


class GraphStep:
    """One bench step (fprop, dgrad, wgrad of every layer) captured into CUDA
    graphs.  An event-record node between two kernels of a graph costs about
    7 us per call here (the step measured 0.632 ms with an event pair around
    each of its 15 calls and 0.526 ms without), so the timed step `g` holds
    the calls alone between the two step events.  `g_pass[kind]` holds the
    five calls of one pass kind alone (per-pass rates and the implicit-GEMM
    launch time), and `g_calls` the step with an event pair around each call
    (the per-layer table, which therefore includes those nodes)."""

    def __init__(self, layers):
        def ev():
            return torch.cuda.Event(enable_timing=True, external=True)
        self.calls = [(kind, L) for L in layers for kind in ("fprop", "dgrad", "wgrad")]

        def capture(calls, per_call):
            g = torch.cuda.CUDAGraph()
            s0, s1 = ev(), ev()
            evs = [(ev(), ev()) for _ in calls] if per_call else None
            with torch.cuda.graph(g):
                s0.record()
                for i, (kind, L) in enumerate(calls):
                    if per_call:
                        evs[i][0].record()
                    getattr(L, kind)()
                    if per_call:
                        evs[i][1].record()
                s1.record()
            g.replay()                     # one untimed replay checks the graph runs
            torch.cuda.synchronize()
            return g, (s0, s1), evs

        self.g, self.ev_step, _ = capture(self.calls, False)
        self.g_calls, self.ev_calls_step, self.ev_calls = capture(self.calls, True)
        self.g_pass = {k: capture([(k, L) for L in layers], False)[:2]
                       for k in ("fprop", "dgrad", "wgrad")}

    def step_ms(self):
        return self.ev_step[0].elapsed_time(self.ev_step[1])

    def pass_ms(self, kind):
        a, b = self.g_pass[kind][1]
        return a.elapsed_time(b)

    def call_ms(self):
        return [(kind, L, a.elapsed_time(b)) for (kind, L), (a, b) in zip(self.calls, self.ev_calls)]


def volume_pass(name, kind, device="cuda"):
    """One pass of a 3D workload as a callable (for --only and ncu captures)."""
    import convolution_implicit_gemm_gb300 as igc
    wl = WORKLOADS[name]
    pb = wl["problem3d"]
    Do, P, Q = igc.conv3d_output_size(pb)
    inp = make_inputs3d(pb, Do, P, Q, wl["dtype"], wl["recipe"], wl["seed"], bias=True)
    X, W, b, dY = (inp[k].to(device) for k in ("X", "W", "bias", "dY"))
    if kind == "fprop":
        Y = torch.empty((pb["N"], Do, P, Q, pb["K"]), dtype=X.dtype, device=device)
        return lambda: igc.conv3d_fprop(pb, X.dtype, X, W, b, None, Y, 1.0, 0.0, True)
    if kind == "dgrad":
        dX = torch.empty_like(X)
        return lambda: igc.conv3d_dgrad(pb, X.dtype, dY, W, None, dX, 1.0, 0.0)
    dW = torch.empty(tuple(W.shape), dtype=torch.float32, device=device)
    need = igc.conv3d_wgrad_workspace_size(pb, X.dtype, torch.float32)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return lambda: igc.conv3d_wgrad(pb, X.dtype, torch.float32, X, dY, None, dW, 1.0, 0.0, ws,
                                    need)


def int8_pass(kind, device="cuda"):
    """One pass of the int8 workload (64 x 56 x 56, 128 -> 128, 3x3) as a
    callable: the requantised forward pass, or the int32 data / weight
    gradient."""
    import convolution_implicit_gemm_gb300 as igc
    wl = WORKLOADS["int8_56x56_128to128_3x3"]
    pb = wl["problem"]
    P, Q = igc.conv2d_output_size(pb)
    inp = make_inputs(pb, P, Q, "i8", "int8", wl["seed"], bias=True)
    X, Wt, b, dY = (inp[k].to(device) for k in ("X", "W", "bias", "dY"))
    if kind == "fprop":
        Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=torch.int8, device=device)
        need = igc.conv2d_fprop_int8_workspace_size(pb)
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        return lambda: igc.conv2d_fprop_int8(pb, X, Wt, b, Y, wl["act_scale"], wl["w_scale"],
                                             wl["out_scale"], True, ws, need)
    if kind == "dgrad":
        dX = torch.empty((pb["N"], pb["H"], pb["W"], pb["C"]), dtype=torch.int32, device=device)
        ws = torch.empty(igc.conv2d_dgrad_int8_workspace_size(pb), dtype=torch.uint8,
                         device=device)
        return lambda: igc.conv2d_dgrad_int8(pb, dY, Wt, dX, ws)
    dW = torch.empty((pb["K"], pb["R"], pb["S"], pb["C"]), dtype=torch.int32, device=device)
    ws = torch.empty(igc.conv2d_wgrad_int8_workspace_size(pb), dtype=torch.uint8, device=device)
    return lambda: igc.conv2d_wgrad_int8(pb, X, dY, dW, ws)


def permute_pass(kind, device="cuda"):
    """The permute of the first sweep layer's activations (128 x 64 x 56 x
    56 bf16), NCHW -> NHWC or back."""
    import convolution_implicit_gemm_gb300 as igc
    pb = WORKLOADS[RESNET50_SWEEP[0]]["problem"]
    N, C, H, W = pb["N"], pb["C"], pb["H"], pb["W"]
    src = torch.randn((N, C, H, W), device=device).to(torch.bfloat16)
    dst = torch.empty((N, H, W, C), dtype=torch.bfloat16, device=device)
    if kind == "nchw_to_nhwc":
        return lambda: igc.nchw_to_nhwc(src, dst, N, C, H, W)
    return lambda: igc.nhwc_to_nchw(dst, src, N, C, H, W)


def run_only(args):
    """One pass of one workload, launched warmup + steps times on cuda:0 (for
    ncu captures: skip `warmup` launches of the kernel, capture the next).
    LAYER:PASS takes the sweep and row workloads (PASS fprop, dgrad, wgrad,
    or winograd for a 3x3 stride-1 layer), int8_56x56_128to128_3x3:PASS the
    int8 passes, permute:nchw_to_nhwc / permute:nhwc_to_nchw the permutes."""
    import convolution_implicit_gemm_gb300 as igc
    igc.load()
    name, kind = args.only.split(":")
    if name == "permute":
        fn = permute_pass(kind)
    elif name == "int8_56x56_128to128_3x3":
        fn = int8_pass(kind)
    elif "problem3d" in WORKLOADS[name]:
        fn = volume_pass(name, kind)
    else:
        L = Layer(name, batch=args.batch)
        if kind == "winograd":
            need = igc.conv2d_fprop_winograd_workspace_size(L.pb, L.td)
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            fn = lambda: igc.conv2d_fprop_winograd(L.pb, L.td, L.X, L.W, L.b, None, L.Y,  # noqa
                                                   1.0, 0.0, L.relu, ws)
        else:
            fn = getattr(L, kind)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = timed_launches(lambda: [fn() for _ in range(args.steps)], torch.cuda.current_stream())
    torch.cuda.synchronize()
    st = igc.igconv_get_device_status()
    if st != 0:
        raise SystemExit(f"device status {igc.igconv_status_string(st)}")
    print(json.dumps({"only": args.only, "launches": args.steps,
                      "ms_per_call": a.elapsed_time(b) / max(1, args.steps)}), flush=True)


def require_device_ok(igc, where):
    """Reads (and clears) the library's device error word after a timed
    region; a kernel that gave up a bounded wait records a code there and
    exits early, which would otherwise show up as a faster time."""
    torch.cuda.synchronize()
    st = igc.igconv_get_device_status()
    if st != 0:
        print(f"bench: device status '{igc.igconv_status_string(st)}' after {where}",
              file=sys.stderr, flush=True)
        raise SystemExit(3)
    return "ok"


FRAC_BITS = {"f16": 10, "bf16": 7}
MIN_NORMAL_EXP = {"f16": -14, "bf16": -126}


def _elem_bound(ref, A, fmt):
    """Per-element bound used by the parity tests: one unit in the last place
    of the output format (fp32: 2^-23 relative) plus 2^-10 of sum |x*w|."""
    import numpy as np
    if fmt == "f32":
        return np.abs(ref) * 2.0 ** -23 + 2.0 ** -10 * A
    ax = np.abs(ref)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, MIN_NORMAL_EXP[fmt])
    return np.ldexp(1.0, (e - FRAC_BITS[fmt]).astype(np.int64)) + 2.0 ** -10 * A


def check_outputs(layers, samples, seed):
    """Compares `samples` seeded elements of each output of every layer (Y,
    dX, dW as the last timed step left them) with the CPU oracle on the same
    inputs.  Run outside every timed region."""
    import numpy as np

    import oracle
    oracle.build()
    worst, count, failed = 0.0, 0, []
    for i, L in enumerate(layers):
        X64 = L.cpu["X"].to(torch.float64).numpy()
        W64 = L.cpu["W"].to(torch.float64).numpy()
        dY64 = L.cpu["dY"].to(torch.float64).numpy()
        b64 = L.cpu["bias"].to(torch.float64).numpy() if L.bias else None
        for kind, out, fmt in (("fprop", L.Y, L.dtype), ("dgrad", L.dX, L.dtype),
                               ("wgrad", L.dW, L.dw_dtype)):
            flat = out.reshape(-1)
            idx = sample_indices(flat.numel(), samples, seed + 31 * i).numpy()
            got = flat[torch.from_numpy(idx).to(flat.device)].to(torch.float64).cpu().numpy()
            if kind == "fprop":
                ref, A = oracle.fprop(L.pb, X64, W64, bias=b64, relu=L.relu, idx=idx,
                                      want_abs=True)
            elif kind == "dgrad":
                ref, A = oracle.dgrad(L.pb, dY64, W64, idx=idx, want_abs=True)
            else:
                ref, A = oracle.wgrad(L.pb, X64, dY64, idx=idx, want_abs=True)
            ratio = float(np.max(np.abs(got - ref) / _elem_bound(ref, A, fmt)))
            if not np.isfinite(got).all() or ratio > 1.0:
                failed.append(f"{L.name}:{kind}")
            worst = max(worst, ratio)
            count += idx.size
    return {"checked": not failed, "samples_per_pass": samples, "elements": count,
            "max_err_over_bound": worst, "failed": failed,
            "bound": "|err_i| <= ulp(out_i) + 2^-10 * sum|x*w|_i against the fp64 oracle"}


def job_rate(step_flops, steps, total_ms, world, device):
    """Whole-job TFLOP/s over all ranks and the time it is taken over: the
    slowest rank's time (max over ranks) and the work of every rank (each
    rank runs the same step on its own GPU: weak scaling)."""
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    total_ms = float(t.item())
    return step_flops * steps * world / (total_ms * 1e-3) / 1e12, total_ms


def run_ours(args, rank, world, local_rank):
    import convolution_implicit_gemm_gb300 as igc
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    igc.load()
    stream = torch.cuda.current_stream()
    layers = [Layer(n, batch=args.batch, device=device) for n in RESNET50_SWEEP]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    step_flops = sum(3 * L.flops for L in layers)

    def step(record=None):
        for L in layers:
            if record is None:
                L.fprop()
                L.dgrad()
                L.wgrad()
            else:
                record.append(("fprop", L, timed_launches(L.fprop, stream)))
                record.append(("dgrad", L, timed_launches(L.dgrad, stream)))
                record.append(("wgrad", L, timed_launches(L.wgrad, stream)))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # The step's 15 calls (20 kernel launches) are captured once into a CUDA
    # graph, with an event pair around every call and around the step, and
    # replayed: launch gaps shrink to the graph's, every kernel still runs
    # in full.  Each replay is read back before the next one reuses the events.
    graph = None
    if not args.no_graph:
        try:
            graph = GraphStep(layers)
        except Exception as exc:  # noqa: BLE001  (capture unsupported: time the stream)
            print(f"graph capture failed ({exc}); timing stream launches", file=sys.stderr)
            graph = None
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.3)
    step_ms, records = [], []
    pass_graph_ms = {"fprop": [], "dgrad": [], "wgrad": []}
    torch.cuda.synchronize()
    for _ in range(args.steps):
        flush.zero_()                      # L2 flushed between timed steps, outside the timing
        if graph is not None:
            graph.g.replay()
            torch.cuda.synchronize()
            step_ms.append(graph.step_ms())
        else:
            rec = []
            a, b = timed_launches(lambda: step(rec), stream)
            torch.cuda.synchronize()
            step_ms.append(a.elapsed_time(b))
            records.append([(kind, L, x.elapsed_time(y)) for kind, L, (x, y) in rec])
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = {"timed_steps": require_device_ok(igc, "the timed steps")}
    if graph is not None:
        # the per-pass graphs and the per-call graph, each from a flushed L2
        for _ in range(min(args.steps, 50)):
            for kind in pass_graph_ms:
                flush.zero_()
                graph.g_pass[kind][0].replay()
                torch.cuda.synchronize()
                pass_graph_ms[kind].append(graph.pass_ms(kind))
            flush.zero_()
            graph.g_calls.replay()
            torch.cuda.synchronize()
            records.append(graph.call_ms())
        status["pass_graphs"] = require_device_ok(igc, "the per-pass graphs")
    check = None
    if rank == 0 and not args.no_check:
        check = check_outputs(layers, args.check_samples, 777)
        if not check["checked"]:
            print(f"bench: outputs differ from the oracle: {check}", file=sys.stderr, flush=True)
            raise SystemExit(4)
    # the same step with L2 left warm between replays (no flush)
    warm_ms, warm_records = [], []
    for _ in range(min(args.steps, 50)):
        if graph is not None:
            graph.g.replay()
            torch.cuda.synchronize()
            warm_ms.append(graph.step_ms())
            graph.g_calls.replay()
            torch.cuda.synchronize()
            warm_records.append(graph.call_ms())
        else:
            rec = []
            a, b = timed_launches(lambda: step(rec), stream)
            torch.cuda.synchronize()
            warm_ms.append(a.elapsed_time(b))
            warm_records.append([(kind, L, x.elapsed_time(y)) for kind, L, (x, y) in rec])
    status["l2_warm_steps"] = require_device_ok(igc, "the L2-warm steps")
    if world > 1:
        torch.distributed.barrier()
    total_ms = sum(step_ms)
    # per-pass and per-kernel accounting
    pass_ms = {"fprop": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    pass_flops = {"fprop": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    gemm_ms, gemm_flops, gemm_launches = 0.0, 0.0, 0
    per_layer = {}
    for rec in records:
        for kind, L, ms in rec:
            pass_ms[kind] += ms
            pass_flops[kind] += L.flops
            per_layer.setdefault(L.name, {}).setdefault(kind, 0.0)
            per_layer[L.name][kind] += ms / len(records)
            if kind in ("fprop", "dgrad"):
                gemm_ms += ms
                gemm_flops += L.flops
                gemm_launches += 1
    gemm_launches //= max(1, len(records))
    if graph is not None:
        # per-pass rates and the implicit-GEMM launch time from the graphs of
        # one pass kind each (no event nodes between their kernels)
        for kind, v in pass_graph_ms.items():
            pass_ms[kind] = sum(v)
            pass_flops[kind] = len(v) * sum(L.flops for L in layers)
        gemm_ms = pass_ms["fprop"] + pass_ms["dgrad"]
        gemm_flops = pass_flops["fprop"] + pass_flops["dgrad"]
    launches_per_step = 4 * len(layers)    # fprop 1, dgrad 1, wgrad 2 (GEMM + reduction)

    # end-to-end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        for L in layers:
            L.make_host()
        pipe = E2EPipeline(layers, stream)
        for _ in range(2):
            pipe.step()
        torch.cuda.synchronize()
        # median over the steps: the host link is shared with the other GPU
        # of the same CPU, so single steps can be slowed by traffic not ours
        e2e_all = []
        for _ in range(max(1, args.e2e_steps)):
            a, b = timed_launches(pipe.step, stream)
            torch.cuda.synchronize()
            e2e_all.append(a.elapsed_time(b))
        e2e_ms = statistics.median(e2e_all)
        status["e2e"] = require_device_ok(igc, "the end-to-end steps")
        e2e = {"value": step_flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(L.h2d for L in layers),
               "d2h_bytes_per_step": sum(L.d2h for L in layers),
               "ms_per_step": e2e_ms, "steps": len(e2e_all),
               "ms_min_max": [min(e2e_all), max(e2e_all)],
               "how": "per layer: pinned H2D copies on one stream (X, W, then dY), each pass "
                      "on a second once its inputs landed, each result's D2H copy on a third as "
                      "soon as its pass is done; layers overlap (smallest input first, "
                      "smallest output last), steps do not",
               "layer_order": [L.name for L in pipe.layers]}

    rows = None
    if not args.no_rows and rank == 0:
        rows = measure_rows(args, device, stream)
        status["rows"] = require_device_ok(igc, "the rows")

    value, total_ms = job_rate(step_flops, args.steps, total_ms, world, device)
    ms_per_step = total_ms / args.steps
    layer_rows = {n: {k: {"us": v * 1e3,
                          "TFLOP/s": next(L.flops for L in layers if L.name == n) / (v * 1e-3) / 1e12}
                      for k, v in d.items()} for n, d in per_layer.items()}
    warm_layers = {}
    for rec in warm_records:
        for kind, L, ms in rec:
            warm_layers.setdefault(L.name, {}).setdefault(kind, 0.0)
            warm_layers[L.name][kind] += ms / len(warm_records)
    l2_warm = None
    if warm_ms:
        wm = sum(warm_ms) / len(warm_ms)
        l2_warm = {"value": step_flops * world / (wm * 1e-3) / 1e12, "ms_per_step": wm,
                   "steps": len(warm_ms),
                   "layers": {n: {k: {"us": v * 1e3,
                                      "TFLOP/s": next(L.flops for L in layers if L.name == n)
                                      / (v * 1e-3) / 1e12}
                                  for k, v in d.items()} for n, d in warm_layers.items()}}
    launch = ("CUDA graph of the step's 15 calls (20 kernels) between two events, replayed "
              "once per step; passes and the roofline from graphs of one pass kind each, the "
              "per-layer table from a graph with an event pair around every call (those "
              "event nodes add a few us per call)"
              if graph is not None else "stream launches")
    return dict(layers=layers, value=value, ms_per_step=ms_per_step, clocks=clk, e2e=e2e,
                status=status, check=check, l2_warm=l2_warm,
                launch=launch,
                layer_rows=layer_rows,
                pass_tflops={k: pass_flops[k] / (pass_ms[k] * 1e-3) / 1e12 for k in pass_ms},
                gemm=(gemm_flops, gemm_ms, gemm_launches), rows=rows,
                launches=launches_per_step * args.steps, step_flops=step_flops)


def time_call(fn, stream, reps=10, warm=3, flush=None):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = timed_launches(fn, stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / reps


def measure_rows(args, device, stream):
    """The other hot-path rows, each timed on its own (L2 flushed between
    repetitions): permutes, the strided / dilated layers, int8 fprop."""
    import convolution_implicit_gemm_gb300 as igc
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    rows = {}
    # T1: permute the first layer's activations NCHW -> NHWC and back
    pb = WORKLOADS[RESNET50_SWEEP[0]]["problem"]
    N, C, H, W = (args.batch or pb["N"]), pb["C"], pb["H"], pb["W"]
    src = torch.randn((N, C, H, W), device=device).to(torch.bfloat16)
    dst = torch.empty((N, H, W, C), dtype=torch.bfloat16, device=device)
    nbytes = 2 * src.numel() * src.element_size()
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # a plain device copy of the same bytes: what one launch of this size can
    # move (launch, ramp-up and tail weigh on a ~20 us kernel; the HBM peak
    # was measured on a 2 GB copy)
    copy_ms = time_call(lambda: dst.view(-1).copy_(src.view(-1)), stream, flush=flush)
    copy_gbs = nbytes / (copy_ms * 1e-3) / 1e9
    # streamed: 8 calls back to back over 4 buffer pairs (4 x 2 x 51 MB, more
    # than the 129 MB L2, so every call reads its source from HBM), the time
    # per call without one launch's ramp-up and tail
    pairs = [(torch.randn((N, C, H, W), device=device).to(torch.bfloat16),
              torch.empty((N, H, W, C), dtype=torch.bfloat16, device=device)) for _ in range(4)]
    for name, fn, many in (
            ("nchw_to_nhwc", lambda: igc.nchw_to_nhwc(src, dst, N, C, H, W),
             lambda: [igc.nchw_to_nhwc(a, b, N, C, H, W) for _ in range(2) for a, b in pairs]),
            ("nhwc_to_nchw", lambda: igc.nhwc_to_nchw(dst, src, N, C, H, W),
             lambda: [igc.nhwc_to_nchw(b, a, N, C, H, W) for _ in range(2) for a, b in pairs])):
        ms = time_call(fn, stream, flush=flush)
        gbs = nbytes / (ms * 1e-3) / 1e9
        ms8 = time_call(many, stream, reps=5, flush=flush) / 8
        gbs8 = nbytes / (ms8 * 1e-3) / 1e9
        rows[name] = {"GB/s": gbs, "ms": ms, "shape": [N, C, H, W], "dtype": "bf16",
                      "bytes": nbytes, "frac_hbm": gbs / hbm, "hbm_gbs": hbm,
                      "hbm_source": peak_src, "copy_same_bytes_GB/s": copy_gbs,
                      "frac_copy_same_bytes": gbs / copy_gbs,
                      "streamed": {"GB/s": gbs8, "ms_per_call": ms8, "frac_hbm": gbs8 / hbm,
                                   "how": "8 calls back to back over 4 buffer pairs "
                                          "(411 MB, more than L2), time / 8"}}
    del src, dst, pairs
    # dgrad/wgrad-heavy layers (dilated and strided), all three passes
    for name in ("dilated_112x112_64to64_3x3_d2", "strided_112x112_64to64_3x3_s2",
                 "cutlass_notebook"):
        L = Layer(name, device=device)
        r = {}
        for kind in ("fprop", "dgrad", "wgrad"):
            ms = time_call(getattr(L, kind), stream, flush=flush)
            r[kind] = {"TFLOP/s": L.flops / (ms * 1e-3) / 1e12, "ms": ms}
        rows[name] = r
        del L
    # the first layer of a CNN (3 input channels): the few-channel paths,
    # their 8-channel copies included in the time
    L = Layer("resnet50_stem_224x224_3to64_7x7_s2", device=device)
    r = {}
    for kind, what in (("fprop", "8-channel pixel and filter copies + GEMM"),
                       ("dgrad", "8-channel filter copy + GEMM to fp32 rows + unpad/cast"),
                       ("wgrad", "8-channel pixel copy + tap-packed GEMM + split reduction")):
        ms = time_call(getattr(L, kind), stream, flush=flush)
        r[kind] = {"TFLOP/s": L.flops / (ms * 1e-3) / 1e12, "ms": ms, "includes": what}
    rows["resnet50_stem_224x224_3to64_7x7_s2"] = r
    del L
    rows.update(measure_depthwise_rows(device, stream, flush))
    # 3D forward convolution (5D im2col implicit GEMM)
    wl = WORKLOADS["r3d_16x56x56_64to64_3x3x3"]
    pb3 = wl["problem3d"]
    Do, P3, Q3 = igc.conv3d_output_size(pb3)
    inp3 = make_inputs3d(pb3, Do, P3, Q3, wl["dtype"], wl["recipe"], wl["seed"], bias=True)
    X3, W3, b3 = inp3["X"].to(device), inp3["W"].to(device), inp3["bias"].to(device)
    Y3 = torch.empty((pb3["N"], Do, P3, Q3, pb3["K"]), dtype=X3.dtype, device=device)
    dY3 = inp3["dY"].to(device)
    dX3 = torch.empty_like(X3)
    dW3 = torch.empty(tuple(W3.shape), dtype=torch.float32, device=device)
    need3 = igc.conv3d_wgrad_workspace_size(pb3, X3.dtype, torch.float32)
    ws3 = torch.empty(max(need3, 16), dtype=torch.uint8, device=device)
    fl3 = 2.0 * pb3["N"] * Do * P3 * Q3 * pb3["K"] * pb3["C"] * pb3["T"] * pb3["R"] * pb3["S"]
    r3 = {}
    for kind, fn in (
            ("fprop", lambda: igc.conv3d_fprop(pb3, X3.dtype, X3, W3, b3, None, Y3, 1.0, 0.0,
                                               True)),
            ("dgrad", lambda: igc.conv3d_dgrad(pb3, X3.dtype, dY3, W3, None, dX3, 1.0, 0.0)),
            ("wgrad", lambda: igc.conv3d_wgrad(pb3, X3.dtype, torch.float32, X3, dY3, None, dW3,
                                               1.0, 0.0, ws3, need3))):
        ms = time_call(fn, stream, flush=flush)
        r3[kind] = {"TFLOP/s": fl3 / (ms * 1e-3) / 1e12, "ms": ms}
    rows["r3d_16x56x56_64to64_3x3x3"] = r3
    del X3, W3, b3, Y3, dY3, dX3, dW3, ws3
    # Winograd F(2x2, 3x3) forward of the 56x56 64->64 3x3 layer (direct-sum
    # FLOPs over time, so the rate compares with the implicit GEMM's)
    L = Layer("resnet50_56x56_64to64_3x3", device=device)
    need_w = igc.conv2d_fprop_winograd_workspace_size(L.pb, L.td)
    ws_w = torch.empty(need_w, dtype=torch.uint8, device=device)
    ms_w = time_call(lambda: igc.conv2d_fprop_winograd(L.pb, L.td, L.X, L.W, L.b, None, L.Y, 1.0,
                                                       0.0, L.relu, ws_w), stream, flush=flush)
    ms_g = time_call(L.fprop, stream, flush=flush)
    rows["winograd_f2x2_3x3_56x56_64to64"] = {
        "winograd": {"TFLOP/s": L.flops / (ms_w * 1e-3) / 1e12, "ms": ms_w,
                     "workspace_MB": need_w / 1e6,
                     "includes": "input and filter transforms, 16 transform-domain GEMMs "
                                 "(one launch), output transform"},
        "implicit_gemm": {"TFLOP/s": L.flops / (ms_g * 1e-3) / 1e12, "ms": ms_g}}
    del L, ws_w
    # int8 quantised fprop (ops counted like FLOPs: 2 per multiply-add)
    wl = WORKLOADS["int8_56x56_128to128_3x3"]
    pb = wl["problem"]
    P, Q = igc.conv2d_output_size(pb)
    inp = make_inputs(pb, P, Q, "i8", "int8", wl["seed"], bias=True)
    X, Wt, b = inp["X"].to(device), inp["W"].to(device), inp["bias"].to(device)
    Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=torch.int8, device=device)
    need = igc.conv2d_fprop_int8_workspace_size(pb)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    fn = lambda: igc.conv2d_fprop_int8(pb, X, Wt, b, Y, wl["act_scale"], wl["w_scale"],  # noqa
                                       wl["out_scale"], True, ws, need)
    ms = time_call(fn, stream, flush=flush)
    r8 = {"fprop": {"TOPS": conv_flops(pb, P, Q) / (ms * 1e-3) / 1e12, "ms": ms,
                    "includes": "int8->fp16 widening + GEMM"}}
    # int8 data and weight gradients of the same layer (int32 results)
    dY8 = inp["dY"].to(device)
    dX8 = torch.empty((pb["N"], pb["H"], pb["W"], pb["C"]), dtype=torch.int32, device=device)
    dW8 = torch.empty((pb["K"], pb["R"], pb["S"], pb["C"]), dtype=torch.int32, device=device)
    del ws
    for kind, need_fn, call in (
            ("dgrad", igc.conv2d_dgrad_int8_workspace_size,
             lambda w8: igc.conv2d_dgrad_int8(pb, dY8, Wt, dX8, w8)),
            ("wgrad", igc.conv2d_wgrad_int8_workspace_size,
             lambda w8: igc.conv2d_wgrad_int8(pb, X, dY8, dW8, w8))):
        w8 = torch.empty(need_fn(pb), dtype=torch.uint8, device=device)
        ms = time_call(lambda: call(w8), stream, flush=flush)
        r8[kind] = {"TOPS": conv_flops(pb, P, Q) / (ms * 1e-3) / 1e12, "ms": ms,
                    "includes": "int8->fp16 widening + GEMM" +
                                (" + int32 split reduction" if kind == "wgrad" else "")}
        del w8
    rows["int8_56x56_128to128_3x3"] = r8
    return rows


def depthwise_bytes(pb, P, Q, dw_elem, groups):
    """Algorithmic HBM bytes of one grouped/depthwise pass: every operand
    read once and every result written once (16-bit activations and
    filter)."""
    x = pb["N"] * pb["H"] * pb["W"] * pb["C"] * 2
    y = pb["N"] * P * Q * pb["K"] * 2
    wn = pb["K"] * pb["R"] * pb["S"] * (pb["C"] // groups)
    return {"fprop": x + y + wn * 2 + pb["K"] * 2,
            "dgrad": y + x + wn * 2,
            "wgrad": x + y + wn * dw_elem}


def measure_depthwise_rows(device, stream, flush):
    """Depthwise (groups = C = K) and grouped (C/groups = 4) layers, all
    three passes, each timed alone with L2 flushed between repetitions,
    against the measured HBM copy bandwidth (the kernels do R*S*C/groups
    fp32 FMAs per 4 bytes of traffic)."""
    import convolution_implicit_gemm_gb300 as igc
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    rows = {}
    for name in GROUPED_SWEEP:
        wl = WORKLOADS[name]
        pb, G = wl["problem"], wl["groups"]
        P, Q = igc.conv2d_output_size(pb)
        cpu = make_inputs(pb, P, Q, wl["dtype"], wl["recipe"], wl["seed"], bias=wl["bias"],
                          dw_dtype=wl["dw_dtype"], groups=G)
        td, tdw = t[wl["dtype"]], t[wl["dw_dtype"]]
        X, Wt, dY = cpu["X"].to(device), cpu["W"].to(device), cpu["dY"].to(device)
        b = cpu["bias"].to(device) if wl["bias"] else None
        Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=td, device=device)
        dX = torch.empty_like(X)
        dW = torch.empty((pb["K"], pb["R"], pb["S"], pb["C"] // G), dtype=tdw, device=device)
        need = igc.conv2d_grouped_wgrad_workspace_size(pb, G, td, tdw)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        fws_need = igc.conv2d_grouped_fprop_workspace_size(pb, G, td)
        fws = torch.empty(max(fws_need, 16), dtype=torch.uint8, device=device)
        calls = {
            # the workspace entry point: tensor cores for group widths 4..64
            "fprop": lambda: igc.conv2d_grouped_fprop_ws(pb, G, td, X, Wt, b, None, Y, 1.0, 0.0,
                                                         wl["relu"], fws),
            "dgrad": lambda: igc.conv2d_grouped_dgrad_ws(pb, G, td, dY, Wt, None, dX, 1.0, 0.0,
                                                         fws),
            "wgrad": lambda: igc.conv2d_grouped_wgrad(pb, G, td, tdw, X, dY, None, dW, 1.0, 0.0,
                                                      ws, need),
        }
        if fws_need:
            # the same layer on the direct (CUDA-core) kernels, for comparison
            calls["fprop_direct"] = lambda: igc.conv2d_grouped_fprop(pb, G, td, X, Wt, b, None, Y,
                                                                     1.0, 0.0, wl["relu"])
            calls["dgrad_direct"] = lambda: igc.conv2d_grouped_dgrad(pb, G, td, dY, Wt, None, dX,
                                                                     1.0, 0.0)
        nbytes = depthwise_bytes(pb, P, Q, torch.finfo(tdw).bits // 8, G)
        nbytes["fprop_direct"] = nbytes["fprop"]
        nbytes["dgrad_direct"] = nbytes["dgrad"]
        r = {}
        for kind, fn in calls.items():
            ms = time_call(fn, stream, flush=flush)
            gbs = nbytes[kind] / (ms * 1e-3) / 1e9
            r[kind] = {"GB/s": gbs, "ms": ms, "bytes": nbytes[kind],
                       "frac_hbm": gbs / hbm,
                       "GFLOP/s": 2.0 * pb["N"] * P * Q * pb["K"] * pb["R"] * pb["S"]
                       * (pb["C"] // G) / (ms * 1e-3) / 1e9}
        r["peak"] = {"hbm_gbs": hbm, "source": src}
        rows[name] = r
        del X, Wt, dY, Y, dX, dW, ws, fws
    return rows


# ---------------------------------------------------------------------------
# the CPU oracle on bounded samples
# ---------------------------------------------------------------------------
def oracle_sample_step(layers_cpu, budget_s, seed):
    """Runs the oracle on a sample of outputs of every pass of every layer,
    sized so the whole call takes about budget_s seconds; returns the nominal
    FLOPs the sample stands for and the seconds it took."""
    import numpy as np

    import oracle
    flops, secs = 0.0, 0.0
    per_pass = budget_s / (3 * len(layers_cpu))
    for i, (pb, inp, P, Q, bias, relu) in enumerate(layers_cpu):
        X64 = inp["X"].to(torch.float64).numpy()
        W64 = inp["W"].to(torch.float64).numpy()
        dY64 = inp["dY"].to(torch.float64).numpy()
        b64 = inp["bias"].to(torch.float64).numpy() if bias else None
        total_flops = conv_flops(pb, P, Q)
        for kind in ("fprop", "dgrad", "wgrad"):
            numel = {"fprop": pb["N"] * P * Q * pb["K"],
                     "dgrad": pb["N"] * pb["H"] * pb["W"] * pb["C"],
                     "wgrad": pb["K"] * pb["R"] * pb["S"] * pb["C"]}[kind]
            per_elem = total_flops / numel
            # calibrate: a small probe, then the sample that fills the budget
            n = 64
            spent = 0.0
            done = 0
            while spent < per_pass and done < numel:
                idx = sample_indices(numel, n, seed + 97 * i + done).numpy()
                t0 = time.perf_counter()
                if kind == "fprop":
                    oracle.fprop(pb, X64, W64, bias=b64, relu=relu, idx=idx)
                elif kind == "dgrad":
                    oracle.dgrad(pb, dY64, W64, idx=idx)
                else:
                    oracle.wgrad(pb, X64, dY64, idx=idx)
                dt = time.perf_counter() - t0
                spent += dt
                done += idx.size
                flops += idx.size * per_elem
                if dt > 0:
                    n = int(min(max(n * 2, 64), max(64, idx.size * (per_pass - spent) / dt)))
            secs += spent
    return flops, secs


def cpu_layers(batch=None):
    out = []
    for name in RESNET50_SWEEP:
        wl = WORKLOADS[name]
        pb = dict(wl["problem"])
        if batch:
            pb["N"] = batch
        P, Q = out_hw(pb)
        inp = make_inputs(pb, P, Q, wl["dtype"], wl["recipe"], wl["seed"], bias=wl.get("bias"))
        out.append((pb, inp, P, Q, wl.get("bias", False), wl.get("relu", False)))
    return out


def cpu_baseline(args):
    import oracle
    oracle.build()
    layers = cpu_layers(args.batch)
    flops, secs = oracle_sample_step(layers, args.cpu_budget, 4242)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"seeded samples of the outputs of fprop, dgrad and wgrad of the five "
                      f"ResNet-50-shaped layers, ~{args.cpu_budget:.0f} s of fp64 oracle work; "
                      f"value = nominal FLOPs the sampled outputs stand for / seconds"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    layers = cpu_layers(args.batch)
    for w in range(args.warmup):
        oracle_sample_step(layers, 0.2, 1000 + w)
    flops, secs = 0.0, 0.0
    for s in range(args.steps):
        f, t = oracle_sample_step(layers, args.ref_step_s, 2000 + s)
        flops += f
        secs += t
    value = flops / secs / 1e12
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                             "cores": oracle.default_threads(),
                             "sample": f"each step: seeded output samples of every pass of the "
                                       f"five layers, ~{args.ref_step_s:.1f} s of fp64 work"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


METRIC = "conv TFLOP/s per pass (fprop/dgrad/wgrad) and % of GB300 dense tensor peak"


def workload_config(args):
    return {"workload": "ResNet-50-shaped layer sweep: batch %d, bf16 NHWC, 56x56 64->64 3x3, "
                        "56x56 64->256 1x1, 28x28 128->128 3x3, 14x14 256->256 3x3, "
                        "7x7 512->512 3x3; fprop (bias+ReLU) + dgrad + wgrad per layer"
                        % (args.batch or 128),
            "global_batch": (args.batch or 128),
            "passes": ["fprop", "dgrad", "wgrad"], "layers": 5,
            "l2": "flushed between timed steps (512 MiB write); the same step with L2 left "
                  "warm is reported under l2_warm",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch (profiling of a small case only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step's calls as plain stream launches instead of a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true",
                    help="skip the sampled oracle check of the last timed step's outputs")
    ap.add_argument("--check-samples", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=3.0)
    ap.add_argument("--only", default=None, metavar="LAYER:PASS",
                    help="profiling aid: run one pass of one workload warmup + steps times "
                         "(e.g. resnet50_56x56_64to256_1x1:fprop) and print its mean time")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and args.steps > 2:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.only:
        run_only(args)
        return

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    peaks, peak_src = load_peaks()
    gemm_flops, gemm_ms, gemm_launches = res["gemm"]
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    # The peak of the regime the step ran in: the burst figure (cuBLAS timed
    # briefly at the maximum clock) when the sampled SM clock stayed at the
    # maximum during the timed steps, else the sustained one (a seconds-long
    # cuBLAS loop under the power cap, at a lower clock).
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    sm_mhz = res["clocks"].get("sm_mhz")
    sm_max = res["clocks"].get("sm_max_mhz") or peaks.get("sm_max_mhz")
    at_max = sm_mhz is not None and bool(sm_max) and sm_mhz >= 0.97 * float(sm_max)
    peak = burst if at_max else sustained
    src_hash = kernel_source_hash()
    traffic = MEASURED_TRAFFIC.get(src_hash)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": "conv_gemm_kernel (fprop + dgrad launches of the step)",
                "peak_kind": "burst" if at_max else "sustained",
                "peak_source": (f"{peak_src} bf16 {'burst (cuBLAS at the maximum clock)' if at_max else 'sustained (cuBLAS loop under the power cap)'}"
                                f"; chosen because the median SM clock during the timed steps "
                                f"was {sm_mhz} MHz against a maximum of {sm_max} MHz"),
                "peak_burst": burst, "frac_burst": achieved / burst,
                "peak_sustained": sustained, "frac_sustained": achieved / sustained,
                "launches_per_step": gemm_launches,
                "kernel_source": src_hash}
    line = {"metric": METRIC, "value": res["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; no dataset or weights)",
            "config": workload_config(args),
            "frac_of_peak": res["value"] / peak,
            "passes": res["pass_tflops"], "layers": res["layer_rows"], "roofline": roofline,
            "clocks": res["clocks"],
            "gpu_launches": res["launches"], "e2e": res["e2e"], "rows": res["rows"],
            "l2_warm": res["l2_warm"], "check": res["check"],
            "device_status": res["status"], "launch": res["launch"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
