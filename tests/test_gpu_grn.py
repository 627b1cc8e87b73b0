"""The multi-horizon GRN heads on the GPU through the C ABI against the GRN
oracle (FP32 tolerance |gpu - ref| <= 1e-5 + 1e-4 |ref| elementwise), the
batch sum bit-exact against the oracle's canonical reduction of the GPU's own
per-sample rows, and the heads chained into the CfC K loop the way the pages'
training step uses them (h_seq in, grad_h as the K loop's per-step upstream
gradient)."""

import numpy as np
import pytest

import recurrent_cell_gb300 as cfc
from oracle import cfc_oracle as co
from oracle import grn_oracle as go
from recurrent_cell_gb300 import workloads as wl

from gpu_common import PARITY_BIAS, CfcRun, assert_close, dev, host, require_gpu, torch_mod

pytestmark = pytest.mark.gpu


class GrnRun:
    def __init__(self, w, inp):
        torch = torch_mod()
        Hd, M, J, R = w.hidden, w.head_mid, w.n_horizons, w.rows
        self.w = w
        self.t = {k: dev(v) for k, v in inp.items()}
        self.N = cfc.cfc_grn_param_length(Hd, M, J)
        assert self.N == go.grn_param_length(Hd, M, J)
        S = cfc.cfc_grn_saved_per_row(M, J)
        assert S == J * (3 * M + 2)
        self.probs = torch.empty(R, J, device="cuda")
        self.saved = torch.empty(R, S, device="cuda")
        self.grad_h = torch.empty(R, Hd, device="cuda")
        self.scratch = torch.empty(w.B, self.N, device="cuda")
        self.grad = torch.empty(self.N, device="cuda")
        self.ws = torch.empty(cfc.cfc_grn_workspace_bytes(w.B, w.K, Hd, M, J), dtype=torch.uint8, device="cuda")

    def step(self, carry=True, h=None):
        w, t = self.w, self.t
        h = t["h"] if h is None else h
        cfc.cfc_grn_forward(h, t["params"], self.probs, self.saved, w.head_mid, w.n_horizons)
        cfc.cfc_grn_backward(h, t["params"], self.probs, self.saved, t["grad_probs"], t["lam"], self.grad_h,
                             self.scratch, self.grad, self.ws, w.B, w.K, w.head_mid, w.n_horizons,
                             grad_h_carry=t["carry"] if carry else None)
        torch_mod().cuda.synchronize()
        return dict(probs=host(self.probs), saved=host(self.saved), grad_h=host(self.grad_h),
                    per_sample=host(self.scratch), grad_params=host(self.grad))


def reference(w, inp, carry=True):
    return go.grn_backward(inp["h"], inp["params"], inp["grad_probs"], inp["lam"], w.B, w.K, w.hidden,
                           w.head_mid, w.n_horizons, grad_h_carry=inp["carry"] if carry else None)


def check(w, got, ref):
    R, M, J = w.rows, w.head_mid, w.n_horizons
    sv = got["saved"]
    JM = J * M
    assert_close(got["probs"], ref["p"], wl.MATH_FP32, f"{w.name}:probs")
    assert_close(sv[:, :JM].reshape(R, J, M), ref["z1"], wl.MATH_FP32, f"{w.name}:z1")
    assert_close(sv[:, JM:2 * JM].reshape(R, J, M), ref["a1"], wl.MATH_FP32, f"{w.name}:a1")
    assert_close(sv[:, 2 * JM:3 * JM].reshape(R, J, M), ref["z2"], wl.MATH_FP32, f"{w.name}:z2")
    assert_close(sv[:, 3 * JM:3 * JM + J], ref["gate"], wl.MATH_FP32, f"{w.name}:gate")
    assert_close(sv[:, 3 * JM + J:], ref["main"], wl.MATH_FP32, f"{w.name}:main")
    assert_close(got["grad_h"], ref["grad_h"], wl.MATH_FP32, f"{w.name}:grad_h")
    assert_close(got["per_sample"], ref["per_sample"], wl.MATH_FP32, f"{w.name}:per_sample")
    assert_close(got["grad_params"], ref["grad_params"], wl.MATH_FP32, f"{w.name}:grad_params")
    # the batch sum is exactly the canonical reduction of the GPU's rows
    np.testing.assert_array_equal(got["grad_params"], co.reduce_axis0(got["per_sample"]))


CASES = [
    wl.GRN_TINY,
    wl.GRN_SMOKE,
    # ragged 32-row tiles, units and columns not multiples of 16 / 32
    wl.GrnWorkload("grn_ragged_B3_K7_132x20x2", B=3, K=7, hidden=132, head_mid=20, n_horizons=2),
    wl.GrnWorkload("grn_min_B1_K1_4x4x1", B=1, K=1, hidden=4, head_mid=4, n_horizons=1),
    wl.GrnWorkload("grn_max_B2_K5_256x64x8", B=2, K=5, hidden=256, head_mid=64, n_horizons=8),
    wl.GrnWorkload("grn_B5_K13_96x36x5", B=5, K=13, hidden=96, head_mid=36, n_horizons=5, seed=7),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_grn_heads_match_oracle(w):
    require_gpu()
    inp = wl.make_grn_inputs(w)
    check(w, GrnRun(w, inp).step(), reference(w, inp))


def test_grn_heads_without_carry():
    require_gpu()
    w = wl.GRN_TINY
    inp = wl.make_grn_inputs(w, seed=2)
    check(w, GrnRun(w, inp).step(carry=False), reference(w, inp, carry=False))


def test_grn_heads_run_to_run_bit_identical():
    require_gpu()
    w = wl.GRN_SMOKE
    r = GrnRun(w, wl.make_grn_inputs(w))
    first = r.step()
    for _ in range(3):
        cur = r.step()
        for k in first:
            np.testing.assert_array_equal(cur[k], first[k])


def test_grn_heads_chained_with_the_kloop():
    """CfC forward -> heads on h_seq -> heads backward -> grad_h as the K loop's
    grad_h_seq -> CfC backward, against the same chain of oracles."""
    require_gpu()
    cw = wl.TINY
    gw = wl.GrnWorkload("grn_on_tiny", B=cw.B, K=cw.K, hidden=cw.n_hid, head_mid=16, n_horizons=3, seed=4)
    cin = wl.make_inputs(cw, bias_scale=PARITY_BIAS)
    gin = wl.make_grn_inputs(gw)
    run = CfcRun(cw, cin)
    run.forward()
    g = GrnRun(gw, gin)
    got_g = g.step(carry=False, h=run.h_seq.reshape(gw.rows, gw.hidden))
    run.backward(y=False, grad_h_seq=g.grad_h.reshape(cw.B, cw.K, cw.n_hid))
    got = run.results()

    fw = co.forward(cin["x"], cin["h0"], cin["W_in"], cin["W_rec"], cin["b"], cin["dt"])
    h_ref = fw["h_seq"].reshape(gw.rows, gw.hidden)
    ref_g = go.grn_backward(h_ref, gin["params"], gin["grad_probs"], gin["lam"], gw.B, gw.K, gw.hidden,
                            gw.head_mid, gw.n_horizons)
    assert_close(got_g["probs"], ref_g["p"], wl.MATH_FP32, "chain:probs")
    assert_close(got_g["grad_h"], ref_g["grad_h"], wl.MATH_FP32, "chain:grad_h")
    assert_close(got_g["grad_params"], ref_g["grad_params"], wl.MATH_FP32, "chain:grad_params")
    ref = co.backward(cin["x"], cin["h0"], cin["W_in"], cin["W_rec"], cin["b"], cin["dt"],
                      grad_h_seq=ref_g["grad_h"].reshape(cw.B, cw.K, cw.n_hid), per_sample=False)
    for k in ("grad_W_in", "grad_W_rec", "grad_b", "grad_h0", "grad_x"):
        assert_close(got[k], ref[k], wl.MATH_FP32, f"chain:{k}")


def test_grn_rejects_unsupported_sizes():
    require_gpu()
    assert cfc.cfc_grn_param_length(130, 64, 5) == 0     # hidden not a multiple of 4
    assert cfc.cfc_grn_param_length(128, 68, 5) == 0     # head_mid above 64
    assert cfc.cfc_grn_param_length(128, 64, 9) == 0     # more than 8 horizons
    assert cfc.cfc_grn_param_length(260, 64, 5) == 0     # hidden above 256
    assert cfc.cfc_grn_param_length(128, 64, 5) == 63375
