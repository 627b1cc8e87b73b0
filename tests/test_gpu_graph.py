"""The whole step (forward + backward, including the weight-gradient contraction
and reduce_axis0) captured once in a CUDA graph through the C ABI and replayed
on new inputs: the calls allocate nothing and never synchronise, so the replay
must give the eager results bit for bit, for every kernel family."""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import workloads as wl

from gpu_common import PARITY_BIAS, CfcRun, assert_close, dev, host, require_gpu, torch_mod

pytestmark = pytest.mark.gpu

CASES = [
    wl.TINY,
    wl.SMOKE,
    wl.MID.with_(name="mid_B96_K32", B=96, K=32),
    wl.LARGE.with_(name="large_B512", B=512),
]


def _graph_of(fn):
    torch = torch_mod()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up on the capture stream's side
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name.split("_")[0] + f"_B{w.B}")
def test_captured_step_replays_bit_exact(w):
    require_gpu()
    torch = torch_mod()
    r = CfcRun(w, wl.make_inputs(w, seed=1, bias_scale=PARITY_BIAS))

    def step():
        r.forward()
        r.backward()

    g = _graph_of(step)
    inp = wl.make_inputs(w, seed=2, bias_scale=PARITY_BIAS)
    r.set_inputs(inp)
    g.replay()
    torch.cuda.synchronize()
    assert cfc.cfc_device_error(clear=True) == 0
    replayed = r.raw()
    got = r.results()

    r.set_inputs(inp)
    step()
    eager = r.raw()
    for a, b in zip(replayed, eager):
        np.testing.assert_array_equal(a, b)

    ref = oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"],
                          mode=w.math, y=inp["y"], per_sample=False)
    for name in ("grad_W_in", "grad_W_rec", "grad_b"):
        assert_close(got[name], ref[name], w.math, f"{w.name} graph {name}")


def test_captured_static_entry_point():
    """cfc_kloop_forward_backward_static (library-owned workspace) under capture."""
    require_gpu()
    torch = torch_mod()
    w = wl.SMOKE.with_(grad_path=wl.GRAD_GEMM)
    inp = wl.make_inputs(w, seed=3, bias_scale=PARITY_BIAS)
    t = {k: dev(inp[k]) for k in ("x", "h0", "W_in", "W_rec", "b", "dt", "y")}
    H, n_in = w.n_hid, w.n_in
    h_seq = torch.empty(w.B, w.K, H, device="cuda")
    gWi = torch.empty(3, H, n_in, device="cuda")
    gWr = torch.empty(3, H, H, device="cuda")
    gb = torch.empty(3, H, device="cuda")

    def step():
        cfc.cfc_kloop_forward_backward_static(t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["dt"],
                                              h_seq, gWi, gWr, gb, y=t["y"], math=w.math)

    g = _graph_of(step)
    inp2 = wl.make_inputs(w, seed=4, bias_scale=PARITY_BIAS)
    for k in t:
        t[k].copy_(dev(inp2[k]))
    g.replay()
    torch.cuda.synchronize()
    rep = [a.cpu().numpy().copy() for a in (h_seq, gWi, gWr, gb)]
    step()
    torch.cuda.synchronize()
    assert cfc.cfc_device_error(clear=True) == 0
    for a, b in zip(rep, (h_seq, gWi, gWr, gb)):
        np.testing.assert_array_equal(a.view(np.uint32), b.cpu().numpy().view(np.uint32))
    ref = oracle.backward(inp2["x"], inp2["h0"], inp2["W_in"], inp2["W_rec"], inp2["b"], inp2["dt"],
                          mode=w.math, y=inp2["y"], per_sample=False)
    assert_close(host(gWr), ref["grad_W_rec"], w.math, "static graph grad_W_rec")
