"""The tau-cell K loop on the GPU through the C ABI against the tau-cell
oracle (FP32 tolerance |gpu - ref| <= 1e-5 + 1e-4 |ref| elementwise)."""

import numpy as np
import pytest

import recurrent_cell_gb300 as cfc
from oracle import tau_oracle as to
from recurrent_cell_gb300 import workloads as wl

from gpu_common import PARITY_BIAS, assert_close, dev, host, require_gpu, torch_mod

pytestmark = pytest.mark.gpu


class TauRun:
    def __init__(self, w, inp):
        torch = torch_mod()
        B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
        self.w = w
        self.t = {k: dev(v) for k, v in inp.items()}
        nbytes = cfc.cfc_tau_kloop_workspace_bytes(B, K, n_in, H)
        assert nbytes > 0
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.h_seq = torch.empty(B, K, H, device="cuda")
        self.gWi = torch.empty(H, n_in, device="cuda")
        self.gWr = torch.empty(H, H, device="cuda")
        self.gb = torch.empty(H, device="cuda")
        self.gtau = torch.empty(H, device="cuda")
        self.gh0 = torch.empty(B, H, device="cuda")
        self.gx = torch.empty(B, K, n_in, device="cuda")
        self.scratch = torch.empty(B, cfc.cfc_tau_per_sample_length(n_in, H), device="cuda")

    def step(self, y=True, grad_h_seq=None, grad_h_last=None):
        t = self.t
        cfc.cfc_tau_kloop_forward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["tau"], t["dt"],
                                  self.h_seq, self.ws)
        cfc.cfc_tau_kloop_backward(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["tau"], t["dt"],
                                   self.h_seq, self.gWi, self.gWr, self.gb, self.gtau, self.scratch, self.ws,
                                   grad_h_seq=grad_h_seq, grad_h_last=grad_h_last,
                                   y=t["y"] if y else None, grad_h0=self.gh0, grad_x=self.gx)
        torch_mod().cuda.synchronize()
        return dict(h_seq=host(self.h_seq), grad_W_in=host(self.gWi), grad_W_rec=host(self.gWr),
                    grad_b=host(self.gb), grad_tau=host(self.gtau), grad_h0=host(self.gh0),
                    grad_x=host(self.gx), per_sample=host(self.scratch))


def check(w, got, ref):
    for k in ("h_seq", "grad_W_in", "grad_W_rec", "grad_b", "grad_tau", "grad_h0", "grad_x", "per_sample"):
        assert_close(got[k], ref[k], wl.MATH_FP32, f"{w.name}:{k}")


CASES = [
    wl.TAU_TINY,
    wl.TAU_SMOKE,
    wl.TAU_SMOKE.with_(name="tau_B7_K5_dt_per_sample", B=7, K=5, dt_per_sample=True),
    wl.Workload("tau_edge_B1_K1", B=1, K=1, n_in=3, n_hid=5),
    wl.Workload("tau_edge_odd_B5_K9", B=5, K=9, n_in=7, n_hid=33, dt_per_sample=True),
    wl.Workload("tau_edge_n_in_wide", B=3, K=4, n_in=200, n_hid=40),
    # gradient rows in shared memory: a thread's share above 64 floats, or
    # more than 512 threads
    wl.Workload("tau_edge_smem_rows", B=3, K=4, n_in=240, n_hid=64),
    wl.Workload("tau_edge_H160", B=3, K=3, n_in=8, n_hid=160, dt_per_sample=True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tau_cell_matches_oracle(w):
    require_gpu()
    inp = wl.make_tau_inputs(w, bias_scale=PARITY_BIAS)
    got = TauRun(w, inp).step()
    ref = to.tau_backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["tau"], inp["dt"],
                          y=inp["y"])
    check(w, got, ref)


def test_tau_cell_upstream_seeds_and_clamped_taus():
    """Per-step and last-state seeds without y; two taus below the clamp get
    exactly zero gradient."""
    require_gpu()
    w = wl.TAU_TINY
    inp = wl.make_tau_inputs(w, seed=3, bias_scale=PARITY_BIAS)
    inp["tau"][[1, 5]] = np.float32(1e-7)
    rng = np.random.default_rng(4)
    gseq = rng.standard_normal((w.B, w.K, w.n_hid)).astype(np.float32)
    glast = rng.standard_normal((w.B, w.n_hid)).astype(np.float32)
    got = TauRun(w, inp).step(y=False, grad_h_seq=dev(gseq), grad_h_last=dev(glast))
    ref = to.tau_backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["tau"], inp["dt"],
                          grad_h_seq=gseq, grad_h_last=glast)
    check(w, got, ref)
    assert got["grad_tau"][1] == 0.0 and got["grad_tau"][5] == 0.0


def test_tau_cell_run_to_run_bit_identical():
    require_gpu()
    w = wl.TAU_SMOKE
    r = TauRun(w, wl.make_tau_inputs(w, bias_scale=PARITY_BIAS))
    first = r.step()
    for _ in range(3):
        cur = r.step()
        for k in first:
            np.testing.assert_array_equal(cur[k], first[k])


def test_tau_cell_rejects_unsupported_sizes():
    require_gpu()
    assert cfc.cfc_tau_kloop_workspace_bytes(4, 8, 64, 300) == 0     # weights + gradient exceed one SM
    assert cfc.cfc_tau_per_sample_length(0, 5) == 0
