"""The C-ABI library builds, loads and exports every symbol that include/cfc.h
declares; host-side logic and argument validation work without a GPU (no
call here reaches a kernel launch)."""

import ctypes
import os
import re

import pytest

import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import build as cfc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cfc.h")

ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_MODE = -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    cfc_build.build()
    return cfc.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("cfc_kloop_forward", "cfc_kloop_backward", "reduce_axis0",
              "cfc_kloop_workspace_bytes", "cfc_per_sample_length", "cfc_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libcfc.so does not export {name}"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_per_sample_length_and_workspace(lib):
    assert cfc.cfc_per_sample_length(64, 128) == 3 * (64 + 128 + 1) * 128 == 74112
    assert cfc.cfc_per_sample_length(128, 256) == 295680
    assert cfc.cfc_per_sample_length(0, 5) == 0
    # scratch path: W^T copy + activations + dA
    B, K, n_in, H = 32, 64, 64, 128
    ws = cfc.cfc_kloop_workspace_bytes(B, K, n_in, H, cfc.MATH_FP32, cfc.GRAD_SCRATCH)
    assert ws >= (n_in + H) * 3 * H * 4 + 2 * B * K * 3 * H * 4
    assert ws % 256 == 0
    gemm = cfc.cfc_kloop_workspace_bytes(B, K, n_in, H, cfc.MATH_FP32, cfc.GRAD_GEMM)
    assert gemm > ws                                    # + split partials
    bf = cfc.cfc_kloop_workspace_bytes(B, K, n_in, H, cfc.MATH_BF16, cfc.GRAD_SCRATCH)
    assert bf < ws                                      # 2-byte W^T and dA
    for bad in [(0, K, n_in, H, 0, 0), (B, 0, n_in, H, 0, 0), (B, K, 0, H, 0, 0),
                (B, K, n_in, 1025, 0, 0), (B, K, 900, 200, 0, 0), (B, K, n_in, H, 3, 0),
                (B, K, n_in, H, 0, 2)]:
        assert cfc.cfc_kloop_workspace_bytes(*bad) == 0


def test_status_strings(lib):
    assert cfc.cfc_status_string(0) == "ok"
    for st in range(-7, 0):
        assert cfc.cfc_status_string(st) not in ("", "unknown status")
    assert cfc.cfc_status_string(42) == "unknown status"


P = 0x100000          # fake, 16-byte-aligned addresses: validation never dereferences


def _fwd(lib, x=P, h0=P, wi=P, wr=P, b=P, dt=P, dts=0, B=4, K=8, n_in=16, H=32, math=0,
         h_seq=P, ws=P, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.cfc_kloop_workspace_bytes(B, K, n_in, H, math, 0) if B > 0 else 0
    return lib.cfc_kloop_forward(x, h0, wi, wr, b, dt, dts, B, K, n_in, H, math, h_seq, ws,
                                 ws_bytes, None)


def test_forward_argument_validation(lib):
    assert _fwd(lib, x=None) == ERR_NULL
    assert _fwd(lib, h_seq=None) == ERR_NULL
    assert _fwd(lib, math=7) == ERR_MODE
    assert _fwd(lib, B=0) == ERR_SHAPE
    assert _fwd(lib, K=-1) == ERR_SHAPE
    assert _fwd(lib, dts=2) == ERR_SHAPE
    assert _fwd(lib, ws=None) == ERR_WORKSPACE
    assert _fwd(lib, ws_bytes=100) == ERR_WORKSPACE
    assert _fwd(lib, x=P + 4) == ERR_ALIGN


def test_backward_argument_validation(lib):
    B, K, n_in, H = 4, 8, 16, 32
    ws_bytes = lib.cfc_kloop_workspace_bytes(B, K, n_in, H, 0, 0)

    def bwd(gseq=None, glast=None, y=P, gwi=P, scratch=P, path=0, ws_bytes=ws_bytes, gx=None):
        return lib.cfc_kloop_backward(P, P, P, P, P, P, 0, B, K, n_in, H, 0, P, gseq, glast, y,
                                      gwi, P, P, None, gx, scratch, path, P, ws_bytes, None)
    assert bwd(y=None) == ERR_NULL                       # no upstream gradient at all
    assert bwd(gwi=None) == ERR_NULL
    assert bwd(scratch=None) == ERR_NULL                 # scratch path needs the scratch
    assert bwd(path=5) == ERR_MODE
    assert bwd(ws_bytes=ws_bytes - 1) == ERR_WORKSPACE
    assert bwd(gx=P + 8) == ERR_ALIGN
    gemm_bytes = lib.cfc_kloop_workspace_bytes(B, K, n_in, H, 0, 1)
    assert bwd(path=1, scratch=None, ws_bytes=gemm_bytes - 256) == ERR_WORKSPACE


def test_reduce_argument_validation(lib):
    assert lib.reduce_axis0(P, 4, 0, P, None) == 0        # nothing to do: no launch
    assert lib.reduce_axis0(P, -1, 10, P, None) == ERR_SHAPE
    assert lib.reduce_axis0(P, 4, -10, P, None) == ERR_SHAPE
    assert lib.reduce_axis0(P, 4, (1 << 35) + 1, P, None) == ERR_SHAPE
    assert lib.reduce_axis0(None, 4, 10, P, None) == ERR_NULL
    assert lib.reduce_axis0(P, 4, 10, None, None) == ERR_NULL
    assert lib.reduce_axis0(P + 2, 4, 10, P, None) == ERR_ALIGN


def test_reduce_multi_argument_validation(lib):
    """Every entry is checked before anything is launched (no GPU needed)."""
    def call(ins, nbs, nts, outs, count=None):
        n = len(ins)
        a_in = (ctypes.c_void_p * max(n, 1))(*ins)
        a_out = (ctypes.c_void_p * max(n, 1))(*outs)
        a_nb = (ctypes.c_int * max(n, 1))(*nbs)
        a_nt = (ctypes.c_longlong * max(n, 1))(*nts)
        return lib.reduce_axis0_multi(a_in, a_nb, a_nt, a_out, n if count is None else count, None)
    assert call([], [], [], []) == 0                                   # nothing to do
    assert call([P], [4], [0], [P]) == 0                               # empty tail: skipped
    assert call([P], [4], [10], [P], count=-1) == ERR_SHAPE
    assert call([P], [4], [10], [P], count=5000) == ERR_SHAPE
    assert lib.reduce_axis0_multi(None, None, None, None, 1, None) == ERR_NULL
    assert call([P, P], [4, -1], [10, 10], [P, P]) == ERR_SHAPE        # second entry bad
    assert call([P, P], [4, 4], [10, (1 << 35) + 1], [P, P]) == ERR_SHAPE
    assert call([P, None], [4, 4], [10, 10], [P, P]) == ERR_NULL
    assert call([P, P], [4, 4], [10, 10], [P, None]) == ERR_NULL
    assert call([P, P + 2], [4, 4], [10, 10], [P, P]) == ERR_ALIGN
    assert call([P, P], [4, 4], [10, 10], [P, P + 1]) == ERR_ALIGN


def test_tau_argument_validation(lib):
    """tau-cell entry points reject bad arguments before launching anything."""
    B, K, n_in, H = 4, 8, 16, 32
    ws = lib.cfc_tau_kloop_workspace_bytes(B, K, n_in, H)
    assert ws >= B * K * H * 4 and ws % 256 == 0
    assert lib.cfc_tau_per_sample_length(n_in, H) == (n_in + H + 2) * H
    assert lib.cfc_tau_kloop_workspace_bytes(B, K, 64, 300) == 0         # exceeds one SM's shared memory
    assert lib.cfc_tau_kloop_workspace_bytes(0, K, n_in, H) == 0

    def fwd(x=P, dt_stride=0, Hh=H, ws_bytes=ws, ws_ptr=P):
        return lib.cfc_tau_kloop_forward(x, P, P, P, P, P, P, dt_stride, B, K, n_in, Hh, P, ws_ptr, ws_bytes, None)
    assert fwd(x=None) == ERR_NULL
    assert fwd(x=P + 4) == ERR_ALIGN
    assert fwd(dt_stride=2) == ERR_SHAPE
    assert fwd(Hh=0) == ERR_SHAPE
    assert fwd(ws_bytes=ws - 1) == ERR_WORKSPACE
    assert fwd(ws_ptr=None) == ERR_WORKSPACE

    def bwd(y=P, gtau=P, scratch=P, gx=None):
        return lib.cfc_tau_kloop_backward(P, P, P, P, P, P, P, 0, B, K, n_in, H, P, None, None, y,
                                          P, P, P, gtau, None, gx, scratch, P, ws, None)
    assert bwd(y=None) == ERR_NULL                        # no upstream gradient
    assert bwd(gtau=None) == ERR_NULL
    assert bwd(scratch=None) == ERR_NULL
    assert bwd(gx=P + 8) == ERR_ALIGN


def test_selftest_timeout_argument_validation(lib):
    assert lib.cfc_selftest_timeout(0, None) == ERR_SHAPE
    assert lib.cfc_selftest_timeout((1 << 20) + 1, None) == ERR_SHAPE


def test_grn_argument_validation(lib):
    """GRN-heads entry points: lengths and argument checks, no launch."""
    from oracle import grn_oracle as go
    for Hd, M, J in ((128, 64, 5), (4, 4, 1), (256, 64, 8), (132, 20, 2)):
        assert lib.cfc_grn_param_length(Hd, M, J) == go.grn_param_length(Hd, M, J)
        assert lib.cfc_grn_saved_per_row(M, J) == J * (3 * M + 2)
    assert lib.cfc_grn_param_length(130, 64, 5) == 0
    assert lib.cfc_grn_param_length(128, 0, 5) == 0
    assert lib.cfc_grn_param_length(128, 64, 0) == 0
    B, K, Hd, M, J = 4, 8, 32, 16, 3
    ws = lib.cfc_grn_workspace_bytes(B, K, Hd, M, J)
    assert ws >= B * K * J * (2 * M + 3) * 4 and ws % 256 == 0
    assert lib.cfc_grn_workspace_bytes(0, K, Hd, M, J) == 0

    def fwd(h=P, rows=B * K, Hh=Hd, probs=P):
        return lib.cfc_grn_forward(h, rows, Hh, M, J, P, probs, P, None)
    assert fwd(rows=0, h=None) == 0                       # nothing to do
    assert fwd(rows=-1) == ERR_SHAPE
    assert fwd(Hh=6) == ERR_SHAPE
    assert fwd(h=None) == ERR_NULL
    assert fwd(probs=P + 4) == ERR_ALIGN

    def bwd(gp=P, lam=P, carry=None, ws_bytes=ws, ws_ptr=P, Bb=B):
        return lib.cfc_grn_backward(P, Bb, K, Hd, M, J, P, P, P, gp, lam, carry, P, P, P, ws_ptr, ws_bytes, None)
    assert bwd(Bb=0) == ERR_SHAPE
    assert bwd(gp=None) == ERR_NULL
    assert bwd(lam=None) == ERR_NULL
    assert bwd(carry=P + 8) == ERR_ALIGN
    assert bwd(ws_bytes=ws - 1) == ERR_WORKSPACE
    assert bwd(ws_ptr=None) == ERR_WORKSPACE


def test_grn_binding_refuses_a_row_count_other_than_B_times_K():
    """The library reads B*K rows of h, probs, saved, grad_probs and grad_h;
    the Python binding checks the row count before it touches the library or
    a device (CPU tensors suffice: the check comes first)."""
    torch = pytest.importorskip("torch")
    h = torch.zeros(10, 8)
    with pytest.raises(ValueError, match="B\\*K"):
        cfc.cfc_grn_backward(h, None, None, None, None, None, None, None, None, None, 4, 3, 4, 1)
    with pytest.raises(ValueError, match="B\\*K"):
        cfc.cfc_grn_backward(h, None, None, None, None, None, None, None, None, None, 0, 10, 4, 1)
