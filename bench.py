#!/usr/bin/env python
"""Benchmark of the batched CfC K-loop (forward + backward through time +
deterministic gradient reduction) on one GB300, printing ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload smoke|tiny|mid|large]
                  [--impl ours|reference] [--no-secondary]

A step is one pass of the whole path over one batch of synthetic input:
cfc_kloop_forward followed by cfc_kloop_backward with the loss seed
0.5*||h_K - y||^2 (which ends in reduce_axis0 of the gradient partials).
Inputs are resident in device memory; L2 is flushed between timed steps by
writing and then reading a 512 MiB buffer (outside the per-step events).  Throughput is
samples*steps per second (B*K / step time).  For N > 1 (torchrun) every rank
runs an independent replica of the workload on its own GPU (there is no
exchange step on this path in a single-GPU deployment), timing is the max
over ranks and the value is the total over ranks.

--impl reference times the CPU oracle (numpy float64) on bounded samples of
the same workload on all of the host's cores: a process pool (spawn start)
of one single-threaded worker per logical CPU, each worker running the oracle
on its own slice of samples.  The GPU line's cpu_baseline reports that
all-cores figure and the single-core one.

The line ends with a compact `gates` object (the throughput workloads mid and
large, and reduce_axis0 at B = 1024): per case the measured time and the
fraction of its roofline, t_roof / t_measured with t_roof = max(flops / tensor
peak, bytes / HBM peak) over the algorithmic work of the whole step.
"""

import os

# The CPU oracle leg is timed single-threaded: pin BLAS threads before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from recurrent_cell_gb300 import workloads as wl  # noqa: E402

METRIC = "CfC K-loop fwd+bwd samples·steps/sec; reduce_axis0 GB/s; % roofline"
UNIT = "samples·steps/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SM_COUNT_NOMINAL = 152          # used only when no device can be queried
FP32_LANES_PER_SM = 128
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    try:
        with open(PEAKS_FILE) as fh:
            p = json.load(fh)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sust=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sust=1700.0,
                    sm_max_mhz=2070.0, source="fallback")


def fp32_alu_peak_tflops(peaks):
    """FFMA peak: SMs (the device's own count) x 128 fp32 lanes x 2 flop x
    maximum SM clock."""
    return peaks["sm_count"] * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


def fp32_alu_peak_source(peaks):
    return f"{peaks['sm_count']} SMs x 128 FFMA lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz"


# ----------------------------------------------------------------------------
# per-kernel algorithmic work (per launch) for the roofline
# ----------------------------------------------------------------------------

TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense TF32 / BF16 tensor throughput


def kernel_work(name, w, n_split):
    """(flops, bytes, flop engine) of one launch of kernel `name` on workload w.

    Algorithmic work: the method's operands read once and its results written
    once.  Per sample-step the path reads x (forward and weight gradient) and
    writes then reads the state history h_seq; the weights, h0, y and the
    outputs are per call.  The saved activations, dA, the weight gradient's
    split partials and the per-sample scratch are this implementation's
    intermediates and are not counted (an implementation may recompute them
    or keep them on chip).  The reducer's own launch counts its [S, N] input,
    which is its operand.
    """
    B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
    Zc, H3, R = n_in + H, 3 * H, w.B * w.K
    s = 2 if w.math == wl.MATH_BF16 else 4
    N = w.N
    engine = "tensor" if (name.endswith("_tc") or "tma" in name) else "alu"
    if name.startswith("cfc_fwd"):
        flops = 2.0 * R * H3 * Zc
        byts = R * n_in * s + B * H * s + H3 * Zc * s + H3 * 4 + R * H * s
        return flops, byts, engine
    if name.startswith("cfc_bwd"):
        # the carry W_rec^T dA per step; the SIMT kernel also forms grad_x
        kc = Zc if name == "cfc_bwd_simt" else H
        flops = 2.0 * R * H3 * kc
        byts = H3 * kc * s + B * H * s + 2 * B * H * 4
        return flops, byts, engine
    if name.startswith("grad_x"):
        return 2.0 * R * H3 * n_in, R * n_in * 4 + H3 * n_in * s, engine
    if name.startswith("wgrad"):
        flops = 2.0 * R * H3 * (Zc + 1)
        byts = R * Zc * s + (Zc + 1) * H3 * 4
        return flops, byts, engine
    if name == "reduce_axis0":
        return 0.0, 4.0 * (n_split * N + N), "alu"
    if name.startswith("prep_w"):
        return 0.0, 2.0 * H3 * Zc * s, "alu"
    return 0.0, 0.0, "alu"


def step_work(w):
    """(flops, bytes) of one whole step (forward, backward without grad_x,
    weight gradient): per sample-step 2*3H*(Zc) + 2*3H*H + 2*3H*(Zc + 1)
    flop and (n_in + H) * s bytes read and written twice (x in the forward
    and the weight gradient, h_seq written and read back), plus the weights
    and the per-sample h0, y and gradient outputs."""
    B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
    Zc, H3, R = n_in + H, 3 * H, B * K
    s = 2 if w.math == wl.MATH_BF16 else 4
    flops = 2.0 * R * H3 * (Zc + H + Zc + 1)
    byts = 2.0 * R * Zc * s + 2 * H3 * Zc * s + B * H * (s + 4) + (Zc + 1) * H3 * 4
    return flops, byts


def tensor_peak(w, peaks, sustained=False):
    """(peak TFLOP/s, source) of the tensor pipe for the workload's mode."""
    bf16 = peaks["bf16_sust"] if sustained else peaks["bf16"]
    kind = "sustained" if sustained else "burst"
    if w.math == wl.MATH_FP32:       # 3xTF32: three TF32 products per fp32 product
        return bf16 * TF32_OVER_BF16 / 3.0, f"{peaks['source']} bf16 {kind} x 1.1/2.25 (TF32) / 3 (3xTF32)"
    if w.math == wl.MATH_TF32:
        return bf16 * TF32_OVER_BF16, f"{peaks['source']} bf16 {kind} x 1.1/2.25 (TF32)"
    return bf16, f"{peaks['source']} bf16 {kind}"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernels, from the ncu captures summarised under profiles/ (smoke at
# its full size; mid and large captured at a quarter of their batch and
# scaled by 4, the units processed -- at that size the kernels' stores stay
# in L2, so these two count the DRAM reads).  Each entry is valid only
# for the sources it was taken from: the second field is the hash of the
# kernel's own file, the shared device headers and the host dispatch
# (KERNEL_FILES, COMMON_FILES) at capture time; any change to one of those
# files makes that kernel's `traffic` null until its capture is repeated.
COMMON_FILES = ("cfc_internal.cuh", "tc_common.cuh", "api.cu")
KERNEL_FILES = {
    "cfc_fwd_cluster": "cfc_cluster.cu",
    "cfc_bwd_cluster": "cfc_cluster.cu",
    "cfc_fwd_tc": "cfc_tc_kloop.cu",
    "cfc_bwd_cluster_tc": "cfc_tc_kloop.cu",
    "cfc_fwd_stream_tc": "cfc_tc_stream.cu",
    "cfc_bwd_tc": "cfc_tc_stream.cu",
    "cfc_fwd_solo_tc": "cfc_tc_solo.cu",
    "cfc_bwd_solo_tc": "cfc_tc_solo.cu",
    "wgrad_tma_3xtf32": "cfc_tc.cu",
    "wgrad_tma_tf32": "cfc_tc.cu",
    "wgrad_tma_tc": "cfc_tc.cu",
}
PROFILED_TRAFFIC = {
    ("smoke", "cfc_fwd_cluster"): (892745, "685fdff94c64622b"),
    ("smoke", "cfc_bwd_cluster"): (3411456, "685fdff94c64622b"),
    ("smoke", "wgrad_tma_3xtf32"): (4786999, "93311003416cba95"),
    ("mid", "cfc_fwd_solo_tc"): (18798738, "bccb9b48ccf1cc45"),
    ("mid", "cfc_bwd_solo_tc"): (102686574, "bccb9b48ccf1cc45"),
    ("mid", "wgrad_tma_tf32"): (151268645, "93311003416cba95"),
    ("large", "cfc_fwd_stream_tc"): (26883291, "2012e14234dc0310"),
    ("large", "cfc_bwd_tc"): (216595602, "2012e14234dc0310"),
    ("large", "wgrad_tma_tc"): (151995977, "93311003416cba95"),
}


def kernel_source_hash(name):
    """Hash of the files kernel `name` is built and dispatched from."""
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "recurrent_cell_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(set(COMMON_FILES + (KERNEL_FILES[name],))):
        h.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(w, name):
    short = {v.name: k for k, v in wl.SHORT_NAMES.items()}.get(w.name)
    entry = PROFILED_TRAFFIC.get((short, name))
    if entry is None or kernel_source_hash(name) != entry[1]:
        return None
    return entry[0]


def roofline_for(name, w, n_split, avg_ms, peaks, sustained=False):
    flops, byts, engine = kernel_work(name, w, n_split)
    t = avg_ms * 1e-3
    if engine == "tensor":
        flop_peak, flop_src = tensor_peak(w, peaks, sustained)
        flop_bound = "tensor"
    else:
        flop_peak = fp32_alu_peak_tflops(peaks)
        flop_src = fp32_alu_peak_source(peaks)
        flop_bound = "alu"
    t_flop = flops / (flop_peak * 1e12) if flops else 0.0
    t_byte = byts / (peaks["hbm"] * 1e9) if byts else 0.0
    traffic = profiled_traffic(w, name)
    extra = dict(traffic=traffic, traffic_over_algorithmic=(traffic / byts if traffic and byts else None),
                 algorithmic_flops_per_launch=flops, algorithmic_bytes_per_launch=byts)
    if t_flop >= t_byte and flops:
        achieved = flops / t / 1e12
        return dict(kernel=name, bound=flop_bound, achieved=achieved, peak=flop_peak, unit="TFLOP/s",
                    frac=achieved / flop_peak, **extra, peak_source=flop_src)
    achieved = byts / t / 1e9
    return dict(kernel=name, bound="hbm", achieved=achieved, peak=peaks["hbm"], unit="GB/s",
                frac=achieved / peaks["hbm"], **extra, peak_source=f"{peaks['source']} hbm_gbs")


def step_roofline(w, ms_step, peaks):
    """Fraction of the whole step's roofline: t_roof / t_measured with
    t_roof = max(step flops / the mode's tensor peak, step bytes / HBM)."""
    flops, byts = step_work(w)
    peak, _ = tensor_peak(w, peaks) if w.math != wl.MATH_FP32 else (fp32_alu_peak_tflops(peaks), "")
    t_roof = max(flops / (peak * 1e12), byts / (peaks["hbm"] * 1e9))
    compute = "tensor" if w.math != wl.MATH_FP32 else "alu"
    return dict(flops=flops, bytes=byts, t_roof_us=t_roof * 1e6, frac=t_roof / (ms_step * 1e-3),
                bound=compute if flops / (peak * 1e12) >= byts / (peaks["hbm"] * 1e9) else "hbm")


# ----------------------------------------------------------------------------
# clocks sampler
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.lines = []
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
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
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[2:6]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None, reasons=sorted(reasons),
                    samples=len(sm))


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

class Packed:
    def __init__(self, buf, views):
        self.buf, self.views = buf, views


def packed_block(torch, specs, device, pin=False):
    """One uint8 block holding tensors (name, dtype, shape) as views, each at a
    256-byte offset (the C ABI wants 16-byte aligned pointers)."""
    offs, off = {}, 0
    for name, dt, shape in specs:
        offs[name] = off
        n = 1
        for d in shape:
            n *= d
        off += (n * torch.empty((), dtype=dt).element_size() + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = {}
    for name, dt, shape in specs:
        n = 1
        for d in shape:
            n *= d
        nb = n * torch.empty((), dtype=dt).element_size()
        views[name] = buf[offs[name]:offs[name] + nb].view(dt).view(shape)
    return Packed(buf, views)


class Path:
    """Device-resident buffers for one workload and the step = fwd + bwd."""

    def __init__(self, w, device):
        import torch
        import recurrent_cell_gb300 as cfc
        self.torch, self.cfc, self.w = torch, cfc, w
        inp = wl.make_inputs(w)
        st = torch.bfloat16 if w.math == wl.MATH_BF16 else torch.float32
        self.st = st
        B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
        f32 = torch.float32
        src = {k: torch.from_numpy(v).to(dtype=(st if k in ("x", "h0", "W_in", "W_rec") else f32))
               for k, v in inp.items()}
        # The inputs live in one pinned host block and one device block, the
        # three gradients in one device block and one pinned host block, each
        # tensor a view at a 256-byte offset: the end-to-end step moves them
        # with one host-to-device and one device-to-host copy.
        in_specs = [(k, v.dtype, tuple(v.shape)) for k, v in src.items()]
        self.in_host = packed_block(torch, in_specs, device="cpu", pin=True)
        for k, v in src.items():
            self.in_host.views[k].copy_(v)
        self.in_dev = packed_block(torch, in_specs, device=device)
        self.in_dev.buf.copy_(self.in_host.buf)
        self.host, self.t = self.in_host.views, self.in_dev.views
        self.ws = torch.empty(cfc.cfc_kloop_workspace_bytes(B, K, n_in, H, w.math, w.grad_path),
                              dtype=torch.uint8, device=device)
        self.h_seq = torch.empty(B, K, H, dtype=st, device=device)
        g_specs = [("gWi", f32, (3, H, n_in)), ("gWr", f32, (3, H, H)), ("gb", f32, (3, H))]
        self.g_dev = packed_block(torch, g_specs, device=device)
        self.g_host = packed_block(torch, g_specs, device="cpu", pin=True)
        self.gWi, self.gWr, self.gb = (self.g_dev.views[k] for k in ("gWi", "gWr", "gb"))
        self.scratch = (torch.empty(B, w.N, device=device) if w.grad_path == wl.GRAD_SCRATCH else None)
        self.h2d_bytes = self.in_host.buf.numel()
        self.d2h_bytes = self.g_host.buf.numel()
        # rows of the gradient partials that reduce_axis0 sums (from the library)
        self.n_split = cfc.cfc_kloop_grad_splits(B, K, n_in, H, w.math, w.grad_path)

    def step(self):
        t, cfc, w = self.t, self.cfc, self.w
        cfc.cfc_kloop_forward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["dt"], self.h_seq,
                              self.ws, math=w.math)
        cfc.cfc_kloop_backward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["dt"], self.h_seq,
                               self.gWi, self.gWr, self.gb, self.ws, y=t["y"],
                               per_sample_scratch=self.scratch, grad_path=w.grad_path, math=w.math)

    def step_e2e(self):
        self.in_dev.buf.copy_(self.in_host.buf, non_blocking=True)
        self.step()
        self.g_host.buf.copy_(self.g_dev.buf, non_blocking=True)


def timed(torch, fn, steps, flush=None):
    """Per-step CUDA-event times (ms) on the current stream; flush between steps."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        if flush is not None:
            flush()
        s.record()
        fn()
        e.record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def compact_kernels(kernels):
    """Per kernel: average device time per launch (us) and launches per step."""
    return {n: dict(avg_us=round(v["avg_ms"] * 1e3, 2), per_step=v["launches_per_step"])
            for n, v in kernels.items()}


def summarize_trace(records, steps):
    per = {}
    for name, ms in records:
        d = per.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += ms
    total = sum(v[1] for v in per.values()) or 1.0
    return {n: dict(launches=v[0], launches_per_step=v[0] / steps, ms_total=v[1],
                    avg_ms=v[1] / v[0], share=v[1] / total) for n, v in per.items()}


def measure_workload(w, steps, warmup, device, peaks, flush, dist_ctx=None, with_e2e=True):
    import torch
    import recurrent_cell_gb300 as cfc
    p = Path(w, device)
    for _ in range(warmup):
        p.step()
    torch.cuda.synchronize()
    if dist_ctx:
        dist_ctx.barrier()
    torch.cuda.synchronize()
    # the timed steps run untraced; the per-kernel breakdown comes from a
    # separate traced pass (event records around every launch)
    ms = timed(torch, p.step, steps, flush)
    torch.cuda.synchronize()
    if dist_ctx:
        dist_ctx.barrier()
    trace_steps = max(3, min(steps, 20))
    cfc.cfc_trace_enable(True)
    timed(torch, p.step, trace_steps, flush)
    records = cfc.cfc_trace_records()
    cfc.cfc_trace_enable(False)
    torch.cuda.synchronize()
    ms_step = sum(ms) / len(ms)
    kernels = summarize_trace(records, trace_steps)
    top = max(kernels, key=lambda n: kernels[n]["ms_total"])
    roof = roofline_for(top, w, p.n_split, kernels[top]["avg_ms"], peaks, sustained=False)
    out = dict(ms_per_step=ms_step, ms_per_step_median=statistics.median(ms), kernels=kernels,
               roofline=roof, gpu_launches=round(len(records) * steps / trace_steps), n_split=p.n_split)
    if with_e2e:
        e2e_steps = max(3, min(steps, 50))
        for _ in range(2):
            p.step_e2e()
        torch.cuda.synchronize()
        ems = timed(torch, p.step_e2e, e2e_steps, flush)
        out["e2e_ms"] = sum(ems) / len(ems)
        out["h2d"] = p.h2d_bytes
        out["d2h"] = p.d2h_bytes
    del p
    torch.cuda.empty_cache()
    return out


def measure_tau(w, steps, warmup, device, peaks, flush):
    """The pages' single-head tau-cell K loop (FP32): forward + backward with
    the y loss seed, per-sample rows summed by reduce_axis0.  Roofline of the
    dominant kernel against the FFMA peak: forward 2 H (n_in + H) flop per
    sample-step; backward 2 H (n_in + H) (gradient rows) + 2 H H (carry)."""
    import torch
    import recurrent_cell_gb300 as cfc
    inp = wl.make_tau_inputs(w)
    t = {k: torch.from_numpy(v).to(device) for k, v in inp.items()}
    B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
    ws = torch.empty(cfc.cfc_tau_kloop_workspace_bytes(B, K, n_in, H), dtype=torch.uint8, device=device)
    h_seq = torch.empty(B, K, H, device=device)
    g = [torch.empty(H, n_in, device=device), torch.empty(H, H, device=device), torch.empty(H, device=device),
         torch.empty(H, device=device)]
    scratch = torch.empty(B, cfc.cfc_tau_per_sample_length(n_in, H), device=device)

    def step():
        cfc.cfc_tau_kloop_forward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["tau"], t["dt"], h_seq, ws)
        cfc.cfc_tau_kloop_backward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["tau"], t["dt"], h_seq,
                                   *g, scratch, ws, y=t["y"])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = timed(torch, step, steps, flush)          # untraced
    cfc.cfc_trace_enable(True)
    timed(torch, step, steps, flush)               # per-kernel breakdown
    records = cfc.cfc_trace_records()
    cfc.cfc_trace_enable(False)
    kernels = summarize_trace(records, steps)
    ms_step = sum(ms) / len(ms)
    Zc = n_in + H
    flops = {"tau_fwd": 2.0 * H * Zc * B * K, "tau_bwd": (2.0 * H * Zc + 2.0 * H * H) * B * K}
    top = max((n for n in kernels if n in flops), key=lambda n: kernels[n]["ms_total"])
    achieved = flops[top] / (kernels[top]["avg_ms"] * 1e-3) / 1e12
    peak = fp32_alu_peak_tflops(peaks)
    return dict(workload=w.name, value=B * K / (ms_step * 1e-3), unit=UNIT, ms_per_step=ms_step,
                kernels=compact_kernels(kernels),
                roofline=dict(kernel=top, bound="alu", achieved=achieved, peak=peak, unit="TFLOP/s",
                              frac=achieved / peak, peak_source=fp32_alu_peak_source(peaks)))


def measure_grn(w, steps, warmup, device, peaks, flush):
    """The multi-horizon GRN heads on every K position (FP32): forward over the
    B*K trunk rows, backward with grad_h_carry, per-sample rows summed by
    reduce_axis0.  Algorithmic flops per row: forward 2 J M (Hd + M) + 2 J (2 M
    + Hd); backward rows 2 J M (M + Hd) (W2^T dz2, W1^T dz1); per-sample
    gradient 2 J M (Hd + M) + 2 J (2 M + Hd) (one FMA per packed element and
    row).  Roofline of the dominant kernel against the FFMA peak."""
    import torch
    import recurrent_cell_gb300 as cfc
    inp = wl.make_grn_inputs(w)
    t = {k: torch.from_numpy(v).to(device) for k, v in inp.items()}
    Hd, M, J, R = w.hidden, w.head_mid, w.n_horizons, w.rows
    N = cfc.cfc_grn_param_length(Hd, M, J)
    probs = torch.empty(R, J, device=device)
    saved = torch.empty(R, cfc.cfc_grn_saved_per_row(M, J), device=device)
    gh = torch.empty(R, Hd, device=device)
    scratch = torch.empty(w.B, N, device=device)
    grad = torch.empty(N, device=device)
    ws = torch.empty(cfc.cfc_grn_workspace_bytes(w.B, w.K, Hd, M, J), dtype=torch.uint8, device=device)

    def step():
        cfc.cfc_grn_forward(t["h"], t["params"], probs, saved, M, J)
        cfc.cfc_grn_backward(t["h"], t["params"], probs, saved, t["grad_probs"], t["lam"], gh, scratch, grad, ws,
                             w.B, w.K, M, J, grad_h_carry=t["carry"])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = timed(torch, step, steps, flush)          # untraced
    cfc.cfc_trace_enable(True)
    timed(torch, step, steps, flush)               # per-kernel breakdown
    records = cfc.cfc_trace_records()
    cfc.cfc_trace_enable(False)
    kernels = summarize_trace(records, steps)
    ms_step = sum(ms) / len(ms)
    flops = {"grn_fwd": (2.0 * J * M * (Hd + M) + 2.0 * J * (2 * M + Hd)) * R,
             "grn_bwd_rows": 2.0 * J * M * (M + Hd) * R,
             "grn_wgrad": 2.0 * N * R}
    top = max((n for n in kernels if n in flops), key=lambda n: kernels[n]["ms_total"])
    achieved = flops[top] / (kernels[top]["avg_ms"] * 1e-3) / 1e12
    peak = fp32_alu_peak_tflops(peaks)
    return dict(workload=w.name, value=R / (ms_step * 1e-3), unit="rows/s", ms_per_step=ms_step,
                kernels=compact_kernels(kernels),
                roofline=dict(kernel=top, bound="alu", achieved=achieved, peak=peak, unit="TFLOP/s",
                              frac=achieved / peak, peak_source=fp32_alu_peak_source(peaks)))


def measure_reduce_multi(steps, device, peaks, flush, B=32, count=17):
    """count reducer calls of one training step (the pages' step makes 17, one
    per scratch buffer) as count single reduce_axis0 launches and as one
    reduce_axis0_multi call; [B, N_i] fp32 ~ N(0, 1), N_i in 4096 .. 20481."""
    import torch
    import recurrent_cell_gb300 as cfc
    Ns = [4096 * (1 + i % 5) + (i % 3) for i in range(count)]
    mats = [torch.from_numpy(wl.make_reduce_input(B, N, seed=1000 + i)).to(device) for i, N in enumerate(Ns)]
    outs = [torch.empty(N, device=device) for N in Ns]

    def singles():
        for a, o in zip(mats, outs):
            cfc.reduce_axis0(a, o)

    def multi():
        cfc.reduce_axis0_multi(mats, outs)

    for _ in range(3):
        singles()
        multi()
    torch.cuda.synchronize()
    t1 = timed(torch, singles, steps, flush)
    t2 = timed(torch, multi, steps, flush)
    byts = 4.0 * sum(B * N + N for N in Ns)
    ms1, ms2 = sum(t1) / len(t1), sum(t2) / len(t2)
    return dict(B=B, count=count, N=Ns, bytes=byts, singles_ms=ms1, multi_ms=ms2,
                multi_GBps=byts / (ms2 * 1e-3) / 1e9, frac_of_hbm=byts / (ms2 * 1e-3) / 1e9 / peaks["hbm"])


def measure_graph(w, steps, device):
    """The same step launched eagerly and replayed from one CUDA graph captured
    through the C ABI (the calls allocate nothing and never synchronise)."""
    import torch
    p = Path(w, device)
    for _ in range(3):
        p.step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        p.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        p.step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    def batch(fn):
        # back to back, no L2 flush: the host's launch rate is part of the time
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / steps

    out = dict(eager_ms=batch(p.step), graph_ms=batch(g.replay), steps=steps,
               timing="back-to-back steps, no L2 flush")
    del g, p
    torch.cuda.empty_cache()
    return out


def measure_reduce(B, N, steps, device, peaks, flush):
    import torch
    import recurrent_cell_gb300 as cfc
    a = torch.from_numpy(wl.make_reduce_input(B, N, seed=B + N)).to(device)
    out = torch.empty(N, device=device)
    for _ in range(3):
        cfc.reduce_axis0(a, out)
    torch.cuda.synchronize()
    ms = timed(torch, lambda: cfc.reduce_axis0(a, out), steps, flush)
    avg = sum(ms) / len(ms)
    gbs = 4.0 * (B * N + N) / (avg * 1e-3) / 1e9
    # context: torch's own column sum of the same matrix, timed the same way
    # (a reference point for a read-bound reduction of this size, not a parity check)
    ref = torch.empty(N, device=device)
    tms = timed(torch, lambda: torch.sum(a, dim=0, out=ref), steps, flush)
    return dict(B=B, N=N, ms=avg, GBps=gbs, frac_of_hbm=gbs / peaks["hbm"],
                torch_sum_dim0_ms=sum(tms) / len(tms))


# ----------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

def oracle_sample_batch(w):
    """Samples per oracle call: the whole batch when small, else a slice
    (samples are independent, so throughput scales with the slice)."""
    return min(w.B, {wl.MATH_FP32: 64}.get(w.math, 128))


def host_cpu():
    """The host the oracle runs on: architecture, logical CPUs, model name
    where /proc/cpuinfo gives one."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model", "hardware")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return dict(arch=platform.machine(), logical_cpus=os.cpu_count(), model=model)


_ORACLE_INPUTS = {}


def _oracle_slice(name, b, offset):
    """One oracle fwd + bwd on samples offset .. offset+b-1 of workload
    `name` (wrapping around the batch); runs in the calling process or in a
    pool worker.  Returns its wall time in seconds."""
    import oracle
    w = wl.WORKLOADS[name]
    inp = _ORACLE_INPUTS.get(name)
    if inp is None:
        inp = _ORACLE_INPUTS[name] = wl.make_inputs(w)
    idx = (offset + np.arange(b)) % w.B
    sl = {k: (v[idx] if k in ("x", "h0", "y") or (k == "dt" and v.size > 1) else v) for k, v in inp.items()}
    t0 = time.perf_counter()
    oracle.backward(sl["x"], sl["h0"], sl["W_in"], sl["W_rec"], sl["b"], sl["dt"], mode=w.math,
                    y=sl["y"], per_sample=(w.grad_path == wl.GRAD_SCRATCH))
    return time.perf_counter() - t0


def time_oracle(w, seconds=10.0, max_reps=None):
    """The oracle on one core (one BLAS thread), repeated for ~seconds."""
    b = oracle_sample_batch(w)
    _oracle_slice(w.name, b, 0)                  # inputs drawn outside the timing
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_slice(w.name, b, 0)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_reps and reps >= max_reps):
            break
    value = reps * b * w.K / el
    return dict(value=value, unit=UNIT, cores=1, kind="oracle", host=host_cpu(),
                sample=f"{reps} x oracle fwd+bwd on {b} of {w.B} samples, K={w.K} "
                       f"({el:.1f} s, numpy float64, 1 BLAS thread)"), el / reps


class OraclePool:
    """One single-threaded oracle worker per logical CPU (spawn start, so it
    is safe after the GPU has been used).  A round gives every worker its own
    slice of b samples (slices at offsets i*b, wrapping around the batch) and
    waits for all of them."""

    def __init__(self, cores=None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.cores = cores or os.cpu_count() or 1
        self.ex = cf.ProcessPoolExecutor(max_workers=self.cores, mp_context=mp.get_context("spawn"))

    def round(self, w, b):
        t0 = time.perf_counter()
        list(self.ex.map(_oracle_slice, [w.name] * self.cores, [b] * self.cores,
                         [i * b for i in range(self.cores)]))
        return time.perf_counter() - t0

    def close(self):
        self.ex.shutdown()


def time_oracle_all_cores(w, seconds=10.0):
    """Throughput of the oracle on all host cores for ~seconds (after one
    untimed round that starts the workers and draws their inputs)."""
    b = oracle_sample_batch(w)
    pool = OraclePool()
    try:
        pool.round(w, b)
        rounds, el = 0, 0.0
        while el < seconds:
            el += pool.round(w, b)
            rounds += 1
    finally:
        pool.close()
    value = rounds * pool.cores * b * w.K / el
    return dict(value=value, unit=UNIT, cores=pool.cores, kind="oracle", host=host_cpu(),
                sample=f"{rounds} rounds x {pool.cores} workers x oracle fwd+bwd on {b} of {w.B} "
                       f"samples, K={w.K} ({el:.1f} s, numpy float64, 1 BLAS thread per worker)")


# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="smoke", choices=sorted(wl.SHORT_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle timing per CPU leg; 0 skips the CPU legs (profiling runs)")
    ap.add_argument("--reduce-only", action="store_true",
                    help="time only the standalone reduce_axis0 cases and the multi-matrix reducer (profiling aid)")
    ap.add_argument("--tau-only", action="store_true",
                    help="time only the tau-cell K loop on the smoke shape (profiling aid)")
    ap.add_argument("--grn-only", action="store_true",
                    help="time only the multi-horizon GRN heads (forward + backward) on the smoke shape")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: run the workload with this many samples instead of its own B "
                         "(the line's config then names the reduced batch)")
    args = ap.parse_args()
    w = wl.SHORT_NAMES[args.workload]
    if args.batch > 0:
        w = w.with_(B=args.batch, name=f"{w.name}_profiled_at_B{args.batch}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        b = oracle_sample_batch(w)
        pool = OraclePool()
        try:
            for _ in range(args.warmup):
                pool.round(w, b)
            per_step = [pool.round(w, b) for _ in range(args.steps)]
        finally:
            pool.close()
        units = pool.cores * b * w.K
        value = units / (sum(per_step) / len(per_step))
        line = dict(impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus,
                    steps=args.steps, warmup=args.warmup,
                    ms_per_step=1e3 * sum(per_step) / len(per_step), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f64",
                    data="synthetic",
                    config=dict(workload=w.name, B=w.B, K=w.K, n_in=w.n_in, n_hid=w.n_hid,
                                math=wl.MATH_NAMES[w.math], sample_batch=b),
                    cpu_baseline=dict(kind="oracle", cores=pool.cores, value=value, unit=UNIT, host=host_cpu(),
                                      sample=f"each step: {pool.cores} workers (one per logical CPU, "
                                             f"1 BLAS thread each), each the oracle fwd+bwd on {b} of "
                                             f"{w.B} samples"),
                    e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
        print(json.dumps(line))
        return 0

    import torch
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dist_ctx = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist_ctx = dist
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    peaks["sm_count"] = torch.cuda.get_device_properties(device).multi_processor_count
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_sink = torch.empty(1, dtype=torch.float32, device=device)

    def flush():
        # Write a buffer larger than L2 (evicts the previous step's lines), then
        # read it back so the L2 ends holding clean lines: the next timed step
        # then pays no write-back of the flush's own dirty lines.
        flush_buf.fill_(1.0)
        torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)

    if args.reduce_only:
        red = [measure_reduce(B, N, args.steps, device, peaks, flush)
               for B in wl.REDUCE_BATCHES for N in wl.REDUCE_TAILS]
        multi = measure_reduce_multi(args.steps, device, peaks, flush)
        print(json.dumps(dict(metric="reduce_axis0 GB/s", unit="GB/s", steps=args.steps,
                              results=red, multi=multi, peak_hbm_gbs=peaks["hbm"])))
        return 0
    if args.tau_only:
        print(json.dumps(measure_tau(wl.TAU_SMOKE, args.steps, args.warmup, device, peaks, flush)))
        return 0
    if args.grn_only:
        print(json.dumps(measure_grn(wl.GRN_SMOKE, args.steps, args.warmup, device, peaks, flush)))
        return 0

    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    sampler = ClockSampler(str(uuid) if uuid else None)
    main_res = measure_workload(w, args.steps, args.warmup, device, peaks, flush, dist_ctx)
    clocks = sampler.stop()

    ms = main_res["ms_per_step"]
    if dist_ctx:
        t = torch.tensor([ms], device=device)
        dist_ctx.all_reduce(t, op=dist_ctx.ReduceOp.MAX)
        ms = float(t.item())
        e = torch.tensor([main_res["e2e_ms"]], device=device)
        dist_ctx.all_reduce(e, op=dist_ctx.ReduceOp.MAX)
        main_res["e2e_ms"] = float(e.item())
    units = w.B * w.K * world
    value = units / (ms * 1e-3)

    secondary = {}
    gates = {}
    cpu = None
    if rank == 0 and not args.no_secondary and world == 1:
        for name in ("mid", "large"):
            ow = wl.SHORT_NAMES[name]
            if name == args.workload:
                r = main_res
            else:
                r = measure_workload(ow, max(5, min(args.steps, 30)), 3, device, peaks, flush, None,
                                     with_e2e=False)
            sr = step_roofline(ow, r["ms_per_step"], peaks)
            secondary[ow.name] = dict(value=ow.B * ow.K / (r["ms_per_step"] * 1e-3), unit=UNIT,
                                      ms_per_step=r["ms_per_step"], step_roofline=sr,
                                      roofline={k: r["roofline"][k] for k in
                                                ("kernel", "bound", "frac", "traffic", "traffic_over_algorithmic")},
                                      kernels=compact_kernels(r["kernels"]))
            gates[name] = dict(value=round(ow.B * ow.K / (r["ms_per_step"] * 1e-3)), unit=UNIT,
                               ms=round(r["ms_per_step"], 4), gflop=round(sr["flops"] / 1e9, 2),
                               mb=round(sr["bytes"] / 1e6, 1), t_roof_us=round(sr["t_roof_us"], 1),
                               bound=sr["bound"], frac=round(sr["frac"], 4), gate=0.60,
                               met=bool(sr["frac"] >= 0.60))
        red = [measure_reduce(B, N, 20, device, peaks, flush)
               for B in wl.REDUCE_BATCHES for N in wl.REDUCE_TAILS]
        secondary["reduce_axis0"] = red
        for rr in red:
            if rr["B"] == 1024:
                gates[f"reduce_B1024_N{rr['N']}"] = dict(
                    value=round(rr["GBps"], 1), unit="GB/s", ms=round(rr["ms"], 4),
                    mb=round(4.0 * (rr["B"] * rr["N"] + rr["N"]) / 1e6, 1), bound="hbm",
                    frac=round(rr["frac_of_hbm"], 4), gate=0.75, met=bool(rr["frac_of_hbm"] >= 0.75))
        secondary["reduce_axis0_multi"] = measure_reduce_multi(20, device, peaks, flush)
        secondary["tau_cell"] = measure_tau(wl.TAU_SMOKE, 30, 3, device, peaks, flush)
        secondary["grn_heads"] = measure_grn(wl.GRN_SMOKE, 30, 3, device, peaks, flush)
        secondary["cuda_graph"] = {wl.SHORT_NAMES[n].name: measure_graph(wl.SHORT_NAMES[n], 50, device)
                                   for n in ("tiny", "smoke")}
    if rank == 0 and world == 1 and args.cpu_seconds > 0 and args.batch == 0:
        one, _ = time_oracle(w, seconds=args.cpu_seconds)
        cpu = time_oracle_all_cores(w, seconds=args.cpu_seconds)
        cpu["single_core"] = dict(value=one["value"], cores=1, sample=one["sample"])
    if rank != 0:
        return 0
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=ms, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype={wl.MATH_FP32: "f32", wl.MATH_TF32: "tf32", wl.MATH_BF16: "bf16"}[w.math],
        data="synthetic",
        config=dict(workload=w.name, B=w.B, K=w.K, n_in=w.n_in, n_hid=w.n_hid,
                    math=wl.MATH_NAMES[w.math],
                    grad_path="scratch+reduce_axis0" if w.grad_path == wl.GRAD_SCRATCH else "gemm+reduce_axis0",
                    l2="flushed between timed steps (512 MiB write + read, outside the step events)",
                    parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        roofline=main_res["roofline"],
        e2e=dict(value=units / (main_res["e2e_ms"] * 1e-3), unit=UNIT,
                 h2d_bytes_per_step=main_res["h2d"], d2h_bytes_per_step=main_res["d2h"]),
        gpu_launches=main_res["gpu_launches"],
        clocks=clocks,
        step_roofline=step_roofline(w, ms, peaks),
        kernels=compact_kernels(main_res["kernels"]),
    )
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if secondary:
        line["secondary"] = secondary
    if gates:
        line["gates"] = gates          # last, so that a tail of the line keeps it
    print(json.dumps(line))
    if dist_ctx:
        dist_ctx.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
