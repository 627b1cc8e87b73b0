"""Python binding of libcfc (the C ABI in include/cfc.h).

The functions below carry the same names as the C entry points and do
argument marshalling only: they check dtypes/devices/shapes of torch tensors,
pass raw device pointers and the current CUDA stream, and raise on a non-zero
status.  All arithmetic runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams.

There is no fallback: if libcfc.so is missing or cannot be loaded, every call
raises.
"""

from __future__ import annotations

import ctypes
import os

from .workloads import (  # noqa: F401
    MATH_FP32, MATH_TF32, MATH_BF16, GRAD_SCRATCH, GRAD_GEMM,
)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcfc.so")

CFC_OK = 0
_lib = None


class CfcError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed with status {status}: {cfc_status_string(status)}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcfc.so (build it first with recurrent_cell_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libcfc.so not found at {path}: run `python -m recurrent_cell_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    lib.cfc_status_string.argtypes = [i32]
    lib.cfc_status_string.restype = ctypes.c_char_p
    lib.cfc_per_sample_length.argtypes = [i32, i32]
    lib.cfc_per_sample_length.restype = i64
    lib.cfc_kloop_workspace_bytes.argtypes = [i32] * 6
    lib.cfc_kloop_workspace_bytes.restype = sz
    lib.cfc_kloop_forward.argtypes = [vp] * 6 + [i32] * 6 + [vp, vp, sz, vp]
    lib.cfc_kloop_forward.restype = i32
    lib.cfc_kloop_backward.argtypes = ([vp] * 6 + [i32] * 6 + [vp] * 4 + [vp] * 5 + [vp, i32]
                                       + [vp, sz, vp])
    lib.cfc_kloop_backward.restype = i32
    lib.reduce_axis0.argtypes = [vp, i32, i64, vp, vp]
    lib.reduce_axis0.restype = i32
    lib.reduce_axis0_multi.argtypes = [vp, vp, vp, vp, i32, vp]
    lib.reduce_axis0_multi.restype = i32
    lib.cfc_tau_per_sample_length.argtypes = [i32, i32]
    lib.cfc_tau_per_sample_length.restype = i64
    lib.cfc_tau_kloop_workspace_bytes.argtypes = [i32] * 4
    lib.cfc_tau_kloop_workspace_bytes.restype = sz
    lib.cfc_tau_kloop_forward.argtypes = [vp] * 7 + [i32] * 5 + [vp, vp, sz, vp]
    lib.cfc_tau_kloop_forward.restype = i32
    lib.cfc_tau_kloop_backward.argtypes = [vp] * 7 + [i32] * 5 + [vp] * 4 + [vp] * 7 + [vp, sz, vp]
    lib.cfc_tau_kloop_backward.restype = i32
    lib.cfc_grn_param_length.argtypes = [i32, i32, i32]
    lib.cfc_grn_param_length.restype = i64
    lib.cfc_grn_saved_per_row.argtypes = [i32, i32]
    lib.cfc_grn_saved_per_row.restype = i64
    lib.cfc_grn_workspace_bytes.argtypes = [i32] * 5
    lib.cfc_grn_workspace_bytes.restype = sz
    lib.cfc_grn_forward.argtypes = [vp, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.cfc_grn_forward.restype = i32
    lib.cfc_grn_backward.argtypes = [vp] + [i32] * 5 + [vp] * 9 + [vp, sz, vp]
    lib.cfc_grn_backward.restype = i32
    lib.cfc_kloop_forward_backward_static.argtypes = [vp] * 6 + [i32] * 6 + [vp] * 3 + [vp] * 6 + [vp]
    lib.cfc_kloop_forward_backward_static.restype = i32
    lib.cfc_kloop_grad_splits.argtypes = [i32] * 6
    lib.cfc_kloop_grad_splits.restype = i32
    lib.cfc_device_error.argtypes = [i32]
    lib.cfc_device_error.restype = i32
    lib.cfc_selftest_timeout.argtypes = [i32, vp]
    lib.cfc_selftest_timeout.restype = i32
    lib.cfc_trace_enable.argtypes = [i32]
    lib.cfc_trace_enable.restype = i32
    lib.cfc_trace_count.argtypes = []
    lib.cfc_trace_count.restype = i32
    lib.cfc_trace_get.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
    lib.cfc_trace_get.restype = i32
    _lib = lib
    return lib


def cfc_status_string(status: int) -> str:
    return load_library().cfc_status_string(int(status)).decode()


def cfc_per_sample_length(n_in: int, n_hid: int) -> int:
    return int(load_library().cfc_per_sample_length(n_in, n_hid))


def cfc_kloop_workspace_bytes(B, K, n_in, n_hid, math, grad_path=GRAD_SCRATCH) -> int:
    return int(load_library().cfc_kloop_workspace_bytes(B, K, n_in, n_hid, math, grad_path))


def cfc_kloop_grad_splits(B, K, n_in, n_hid, math, grad_path=GRAD_SCRATCH) -> int:
    return int(load_library().cfc_kloop_grad_splits(B, K, n_in, n_hid, math, grad_path))


def cfc_device_error(clear: bool = False) -> int:
    """0 unless a kernel reported a device-side error (waits for the device)."""
    return int(load_library().cfc_device_error(1 if clear else 0))


def cfc_selftest_timeout(max_polls: int = 1000, stream=None) -> None:
    """Run one bounded wait that runs out (see include/cfc.h); afterwards
    cfc_device_error() reports 1 until cleared."""
    _check("cfc_selftest_timeout", load_library().cfc_selftest_timeout(int(max_polls), _stream(stream)))


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, name, dtype=None, shape=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _storage_dtype(math):
    torch = _torch()
    return torch.bfloat16 if math == MATH_BF16 else torch.float32


def _check(fn, status):
    if status != CFC_OK:
        raise CfcError(fn, status)


def cfc_kloop_forward(x, h0, W_in, W_rec, b, dt, h_seq, workspace, math=MATH_FP32, stream=None):
    """Forward K-loop: writes h_seq [B, K, n_hid] and the saved activations in
    ``workspace`` (a uint8 CUDA tensor of cfc_kloop_workspace_bytes bytes)."""
    torch = _torch()
    B, K, n_in = x.shape
    H = h0.shape[1]
    st = _storage_dtype(math)
    f32 = torch.float32
    dt_stride = 0 if dt.numel() == 1 else 1
    status = load_library().cfc_kloop_forward(
        _ptr(x, "x", st, (B, K, n_in)), _ptr(h0, "h0", st, (B, H)),
        _ptr(W_in, "W_in", st, (3, H, n_in)), _ptr(W_rec, "W_rec", st, (3, H, H)),
        _ptr(b, "b", f32, (3, H)), _ptr(dt, "dt", f32, (B,) if dt_stride else None),
        dt_stride, B, K, n_in, H, math,
        _ptr(h_seq, "h_seq", st, (B, K, H)), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream))
    _check("cfc_kloop_forward", status)


def cfc_kloop_backward(x, h0, W_in, W_rec, b, dt, h_seq, grad_W_in, grad_W_rec, grad_b,
                       workspace, grad_h_seq=None, grad_h_last=None, y=None, grad_h0=None,
                       grad_x=None, per_sample_scratch=None, grad_path=GRAD_SCRATCH,
                       math=MATH_FP32, stream=None):
    """Backward through the K loop of the forward that filled ``workspace``."""
    torch = _torch()
    B, K, n_in = x.shape
    H = h0.shape[1]
    st = _storage_dtype(math)
    f32 = torch.float32
    N = 3 * (n_in + H + 1) * H
    dt_stride = 0 if dt.numel() == 1 else 1
    status = load_library().cfc_kloop_backward(
        _ptr(x, "x", st, (B, K, n_in)), _ptr(h0, "h0", st, (B, H)),
        _ptr(W_in, "W_in", st, (3, H, n_in)), _ptr(W_rec, "W_rec", st, (3, H, H)),
        _ptr(b, "b", f32, (3, H)), _ptr(dt, "dt", f32, (B,) if dt_stride else None),
        dt_stride, B, K, n_in, H, math,
        _ptr(h_seq, "h_seq", st, (B, K, H)),
        _ptr(grad_h_seq, "grad_h_seq", f32, (B, K, H), optional=True),
        _ptr(grad_h_last, "grad_h_last", f32, (B, H), optional=True),
        _ptr(y, "y", f32, (B, H), optional=True),
        _ptr(grad_W_in, "grad_W_in", f32, (3, H, n_in)),
        _ptr(grad_W_rec, "grad_W_rec", f32, (3, H, H)),
        _ptr(grad_b, "grad_b", f32, (3, H)),
        _ptr(grad_h0, "grad_h0", f32, (B, H), optional=True),
        _ptr(grad_x, "grad_x", f32, (B, K, n_in), optional=True),
        _ptr(per_sample_scratch, "per_sample_scratch", f32, (B, N),
             optional=(grad_path != GRAD_SCRATCH)),
        grad_path, _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check("cfc_kloop_backward", status)


def reduce_axis0(per_batch, out, stream=None):
    """out[N] = column sums of per_batch[B, N] (overwrite, canonical order)."""
    torch = _torch()
    B, N = per_batch.shape
    status = load_library().reduce_axis0(
        _ptr(per_batch, "per_batch", torch.float32), B, N,
        _ptr(out, "out", torch.float32, (N,)), _stream(stream))
    _check("reduce_axis0", status)


def cfc_grn_param_length(hidden: int, head_mid: int, n_horizons: int) -> int:
    return int(load_library().cfc_grn_param_length(hidden, head_mid, n_horizons))


def cfc_grn_saved_per_row(head_mid: int, n_horizons: int) -> int:
    return int(load_library().cfc_grn_saved_per_row(head_mid, n_horizons))


def cfc_grn_workspace_bytes(B: int, K: int, hidden: int, head_mid: int, n_horizons: int) -> int:
    return int(load_library().cfc_grn_workspace_bytes(B, K, hidden, head_mid, n_horizons))


def cfc_grn_forward(h, params, probs, saved, head_mid: int, n_horizons: int, stream=None):
    """GRN heads forward over the rows of h [R, hidden] (float32): probs
    [R, n_horizons] and the saved intermediates [R, cfc_grn_saved_per_row]."""
    torch = _torch()
    f32 = torch.float32
    R, Hd = h.shape
    N = cfc_grn_param_length(Hd, head_mid, n_horizons)
    S = cfc_grn_saved_per_row(head_mid, n_horizons)
    status = load_library().cfc_grn_forward(
        _ptr(h, "h", f32, (R, Hd)), R, Hd, head_mid, n_horizons, _ptr(params, "params", f32, (N,)),
        _ptr(probs, "probs", f32, (R, n_horizons)), _ptr(saved, "saved", f32, (R, S)), _stream(stream))
    _check("cfc_grn_forward", status)


def cfc_grn_backward(h, params, probs, saved, grad_probs, lam, grad_h, per_sample_scratch, grad_params, workspace,
                     B: int, K: int, head_mid: int, n_horizons: int, grad_h_carry=None, stream=None):
    """GRN heads backward for h [B*K, hidden] rows (r = b*K + k): grad_h,
    the per-sample gradient rows and their batch sum (packed parameter order)."""
    R, Hd = h.shape
    if B < 1 or K < 1 or R != B * K:
        # the library reads B*K rows of every per-row tensor: a mismatch would
        # read past the tensors, so it is refused here
        raise ValueError(f"h has {R} rows; cfc_grn_backward needs B*K = {B}*{K} rows")
    torch = _torch()
    f32 = torch.float32
    N = cfc_grn_param_length(Hd, head_mid, n_horizons)
    S = cfc_grn_saved_per_row(head_mid, n_horizons)
    J = n_horizons
    status = load_library().cfc_grn_backward(
        _ptr(h, "h", f32, (R, Hd)), B, K, Hd, head_mid, J, _ptr(params, "params", f32, (N,)),
        _ptr(probs, "probs", f32, (R, J)), _ptr(saved, "saved", f32, (R, S)),
        _ptr(grad_probs, "grad_probs", f32, (R, J)), _ptr(lam, "lambda", f32, (J,)),
        _ptr(grad_h_carry, "grad_h_carry", f32, (R, Hd), optional=True), _ptr(grad_h, "grad_h", f32, (R, Hd)),
        _ptr(per_sample_scratch, "per_sample_scratch", f32, (B, N)), _ptr(grad_params, "grad_params", f32, (N,)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check("cfc_grn_backward", status)


def cfc_tau_per_sample_length(n_in: int, n_hid: int) -> int:
    return int(load_library().cfc_tau_per_sample_length(n_in, n_hid))


def cfc_tau_kloop_workspace_bytes(B: int, K: int, n_in: int, n_hid: int) -> int:
    return int(load_library().cfc_tau_kloop_workspace_bytes(B, K, n_in, n_hid))


def cfc_tau_kloop_forward(x, h0, W_in, W_rec, b, tau, dt, h_seq, workspace, stream=None):
    """tau-cell forward K loop (float32): writes h_seq [B, K, n_hid] and the
    saved activations in ``workspace``."""
    torch = _torch()
    f32 = torch.float32
    B, K, n_in = x.shape
    H = h0.shape[1]
    dt_stride = 0 if dt.numel() == 1 else 1
    status = load_library().cfc_tau_kloop_forward(
        _ptr(x, "x", f32, (B, K, n_in)), _ptr(h0, "h0", f32, (B, H)), _ptr(W_in, "W_in", f32, (H, n_in)),
        _ptr(W_rec, "W_rec", f32, (H, H)), _ptr(b, "b", f32, (H,)), _ptr(tau, "tau", f32, (H,)),
        _ptr(dt, "dt", f32, (B,) if dt_stride else None), dt_stride, B, K, n_in, H,
        _ptr(h_seq, "h_seq", f32, (B, K, H)), _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check("cfc_tau_kloop_forward", status)


def cfc_tau_kloop_backward(x, h0, W_in, W_rec, b, tau, dt, h_seq, grad_W_in, grad_W_rec, grad_b, grad_tau,
                           per_sample_scratch, workspace, grad_h_seq=None, grad_h_last=None, y=None,
                           grad_h0=None, grad_x=None, stream=None):
    """Backward through the tau-cell K loop of the forward that filled ``workspace``."""
    torch = _torch()
    f32 = torch.float32
    B, K, n_in = x.shape
    H = h0.shape[1]
    N = (n_in + H + 2) * H
    dt_stride = 0 if dt.numel() == 1 else 1
    status = load_library().cfc_tau_kloop_backward(
        _ptr(x, "x", f32, (B, K, n_in)), _ptr(h0, "h0", f32, (B, H)), _ptr(W_in, "W_in", f32, (H, n_in)),
        _ptr(W_rec, "W_rec", f32, (H, H)), _ptr(b, "b", f32, (H,)), _ptr(tau, "tau", f32, (H,)),
        _ptr(dt, "dt", f32, (B,) if dt_stride else None), dt_stride, B, K, n_in, H,
        _ptr(h_seq, "h_seq", f32, (B, K, H)),
        _ptr(grad_h_seq, "grad_h_seq", f32, (B, K, H), optional=True),
        _ptr(grad_h_last, "grad_h_last", f32, (B, H), optional=True),
        _ptr(y, "y", f32, (B, H), optional=True),
        _ptr(grad_W_in, "grad_W_in", f32, (H, n_in)), _ptr(grad_W_rec, "grad_W_rec", f32, (H, H)),
        _ptr(grad_b, "grad_b", f32, (H,)), _ptr(grad_tau, "grad_tau", f32, (H,)),
        _ptr(grad_h0, "grad_h0", f32, (B, H), optional=True),
        _ptr(grad_x, "grad_x", f32, (B, K, n_in), optional=True),
        _ptr(per_sample_scratch, "per_sample_scratch", f32, (B, N)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check("cfc_tau_kloop_backward", status)


def reduce_axis0_multi(per_batch, out, stream=None):
    """out[i][N_i] = column sums of per_batch[i][B_i, N_i] for every i, in few
    launches; the same bits as reduce_axis0 on each pair."""
    torch = _torch()
    per_batch, out = list(per_batch), list(out)
    if len(per_batch) != len(out):
        raise ValueError("per_batch and out must have the same length")
    n = len(per_batch)
    ins = (ctypes.c_void_p * max(n, 1))()
    outs = (ctypes.c_void_p * max(n, 1))()
    nb = (ctypes.c_int * max(n, 1))()
    nt = (ctypes.c_longlong * max(n, 1))()
    for i, (a, o) in enumerate(zip(per_batch, out)):
        if a.dim() != 2:
            raise ValueError(f"per_batch[{i}] must be 2-D")
        B, N = a.shape
        ins[i] = _ptr(a, f"per_batch[{i}]", torch.float32)
        outs[i] = _ptr(o, f"out[{i}]", torch.float32, (N,))
        nb[i], nt[i] = B, N
    status = load_library().reduce_axis0_multi(ins, nb, nt, outs, n, _stream(stream))
    _check("reduce_axis0_multi", status)


def cfc_kloop_forward_backward_static(x, h0, W_in, W_rec, b, dt, h_seq, grad_W_in, grad_W_rec,
                                      grad_b, grad_h_seq=None, grad_h_last=None, y=None,
                                      grad_h0=None, grad_x=None, math=MATH_FP32, stream=None):
    """Forward + backward with the library's fixed internal workspace, for
    callers that cannot allocate device memory.  Computes what
    cfc_kloop_forward + cfc_kloop_backward(grad_path=GRAD_GEMM) compute, always
    on the CUDA-core (SIMT) kernels, so the results agree with those calls
    within the parity tolerances, not bit for bit."""
    torch = _torch()
    B, K, n_in = x.shape
    H = h0.shape[1]
    st = _storage_dtype(math)
    f32 = torch.float32
    dt_stride = 0 if dt.numel() == 1 else 1
    status = load_library().cfc_kloop_forward_backward_static(
        _ptr(x, "x", st, (B, K, n_in)), _ptr(h0, "h0", st, (B, H)),
        _ptr(W_in, "W_in", st, (3, H, n_in)), _ptr(W_rec, "W_rec", st, (3, H, H)),
        _ptr(b, "b", f32, (3, H)), _ptr(dt, "dt", f32, (B,) if dt_stride else None),
        dt_stride, B, K, n_in, H, math,
        _ptr(grad_h_seq, "grad_h_seq", f32, (B, K, H), optional=True),
        _ptr(grad_h_last, "grad_h_last", f32, (B, H), optional=True),
        _ptr(y, "y", f32, (B, H), optional=True),
        _ptr(h_seq, "h_seq", st, (B, K, H)),
        _ptr(grad_W_in, "grad_W_in", f32, (3, H, n_in)),
        _ptr(grad_W_rec, "grad_W_rec", f32, (3, H, H)),
        _ptr(grad_b, "grad_b", f32, (3, H)),
        _ptr(grad_h0, "grad_h0", f32, (B, H), optional=True),
        _ptr(grad_x, "grad_x", f32, (B, K, n_in), optional=True),
        _stream(stream))
    _check("cfc_kloop_forward_backward_static", status)


def cfc_trace_enable(on: bool) -> None:
    """Start (clearing old records) or stop per-kernel event tracing."""
    _check("cfc_trace_enable", load_library().cfc_trace_enable(1 if on else 0))


def cfc_trace_records() -> list:
    """[(kernel name, device milliseconds)] for every traced launch."""
    lib = load_library()
    out = []
    for i in range(lib.cfc_trace_count()):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check("cfc_trace_get", lib.cfc_trace_get(i, ctypes.byref(name), ctypes.byref(ms)))
        out.append((name.value.decode(), float(ms.value)))
    return out
