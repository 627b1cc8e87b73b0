"""Data-parallel step on one GPU: the batch is cut into G contiguous slices, each
slice runs forward + backward through the C ABI with its gradient written
straight into row r of a packed [G, N] buffer (the layout the cross-rank
all_gather produces), and reduce_axis0 sums the rows.  The result must match
the oracle's full-batch gradient within the mode's tolerance and be
bit-identical from run to run."""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import dp
from recurrent_cell_gb300 import workloads as wl

from gpu_common import PARITY_BIAS, assert_close, dev, host, require_gpu, torch_mod

pytestmark = pytest.mark.gpu

CASES = [
    (wl.SMOKE, 3),
    (wl.MID.with_(name="mid_B96", B=96), 2),
    (wl.LARGE.with_(name="large_B256", B=256), 4),
    (wl.LARGE.with_(name="large_B250_ragged", B=250), 3),
]


def _sharded_step(w, inp, G):
    """Returns the [G, N] per-slice gradients and their reduce_axis0 sum."""
    torch = torch_mod()
    st = torch.bfloat16 if w.math == wl.MATH_BF16 else torch.float32
    W_in, W_rec = dev(inp["W_in"], st), dev(inp["W_rec"], st)
    b = dev(inp["b"], torch.float32)
    gathered = torch.empty(G, w.N, device="cuda")
    for r in range(G):
        lo, hi = dp.shard_bounds(w.B, r, G)
        Bs = hi - lo
        x, h0 = dev(inp["x"][lo:hi], st), dev(inp["h0"][lo:hi], st)
        y = dev(inp["y"][lo:hi], torch.float32)
        dt = dev(inp["dt"][lo:hi] if w.dt_per_sample else inp["dt"], torch.float32)
        ws = torch.empty(cfc.cfc_kloop_workspace_bytes(Bs, w.K, w.n_in, w.n_hid, w.math,
                                                       w.grad_path), dtype=torch.uint8,
                         device="cuda")
        h_seq = torch.empty(Bs, w.K, w.n_hid, dtype=st, device="cuda")
        gWi, gWr, gb = dp.gradient_views(gathered[r], w.n_in, w.n_hid)
        scratch = (torch.empty(Bs, w.N, device="cuda") if w.grad_path == wl.GRAD_SCRATCH
                   else None)
        cfc.cfc_kloop_forward(x, h0, W_in, W_rec, b, dt, h_seq, ws, math=w.math)
        cfc.cfc_kloop_backward(x, h0, W_in, W_rec, b, dt, h_seq, gWi, gWr, gb, ws, y=y,
                               per_sample_scratch=scratch, grad_path=w.grad_path, math=w.math)
    out = torch.empty(w.N, device="cuda")
    cfc.reduce_axis0(gathered, out)
    torch.cuda.synchronize()
    assert cfc.cfc_device_error(clear=True) == 0
    return gathered, out


@pytest.mark.parametrize("w, G", CASES, ids=[f"{w.name}_G{G}" for w, G in CASES])
def test_sharded_gradient_matches_full_batch(w, G):
    require_gpu()
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    gathered, out = _sharded_step(w, inp, G)
    # the device reduction of the gathered rows is the canonical order, bit for bit
    rows = gathered.cpu().numpy()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                  oracle.reduce_axis0(rows).view(np.uint32))
    ref = oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"],
                          mode=w.math, y=inp["y"], per_sample=False)
    gWi, gWr, gb = dp.gradient_views(out, w.n_in, w.n_hid)
    for name, got in (("grad_W_in", gWi), ("grad_W_rec", gWr), ("grad_b", gb)):
        assert_close(host(got), ref[name], w.math, f"{w.name} G={G} {name}")
    # run to run
    _, again = _sharded_step(w, inp, G)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                  again.cpu().numpy().view(np.uint32))

