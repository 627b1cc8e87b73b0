"""cfc_kloop_forward_backward_static: the entry point for callers that cannot
allocate device memory while they run the K loop (for example code that runs
under an allocator it does not own, or a plugin that may not call cudaMalloc).
It keeps its workspace in a fixed array inside the library.

It always runs the CUDA-core (SIMT) kernels, so it is checked through the C
ABI against both the oracle and the regular entry points (forward, then
backward with the GEMM gradient path and a caller-allocated workspace, which
run the cluster or tensor-core kernels), with the tolerances of the other
parity tests, in every precision mode, on two calls in a row with different
inputs, so that anything a call left behind in the shared array would show
up in the second call.  This file is collected last on purpose.
"""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import workloads as wl
from gpu_common import PARITY_BIAS, CfcRun, assert_close, host, require_gpu, torch_mod

pytestmark = pytest.mark.gpu

CASES = [
    wl.SMOKE,
    wl.Workload("static_tf32_B37_K5_odd", B=37, K=5, n_in=23, n_hid=40, math=wl.MATH_TF32,
                dt_per_sample=True),
    wl.Workload("static_bf16_B37_K5", B=37, K=5, n_in=24, n_hid=40, math=wl.MATH_BF16,
                dt_per_sample=True),
]
OUTPUTS = ("h_seq", "grad_W_in", "grad_W_rec", "grad_b", "grad_h0", "grad_x")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_static(w, inp):
    torch = torch_mod()
    r = CfcRun(w, inp, grad_path=wl.GRAD_GEMM)      # device copies of the inputs
    t = r.t
    out = dict(h_seq=torch.full_like(r.h_seq, float("nan")),
               grad_W_in=torch.full_like(r.gWi, float("nan")),
               grad_W_rec=torch.full_like(r.gWr, float("nan")),
               grad_b=torch.full_like(r.gb, float("nan")),
               grad_h0=torch.full_like(r.gh0, float("nan")),
               grad_x=torch.full_like(r.gx, float("nan")))
    cfc.cfc_kloop_forward_backward_static(
        t["x"], t["h0"], t["W_in"], t["W_rec"], t["b"], t["dt"], out["h_seq"], out["grad_W_in"],
        out["grad_W_rec"], out["grad_b"], y=t["y"], grad_h0=out["grad_h0"], grad_x=out["grad_x"],
        math=w.math)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}


def run_regular(w, inp):
    r = CfcRun(w, inp, grad_path=wl.GRAD_GEMM)
    r.forward()
    r.backward()
    return r.results()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_workspace_matches_oracle_and_regular_entry_points_twice(w):
    for seed in (101, 202):                      # two calls in a row, different inputs
        inp = wl.make_inputs(w, seed=seed, bias_scale=PARITY_BIAS)
        got = run_static(w, inp)
        want = run_regular(w, inp)
        ref = oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"],
                              mode=w.math, per_sample=False, y=inp["y"])
        for k in OUTPUTS:
            bf = (k == "h_seq" and w.math == wl.MATH_BF16)
            assert_close(got[k], ref[k], w.math, f"{w.name} seed {seed} vs oracle: {k}", state_bf16=bf)
            assert_close(got[k], want[k], w.math, f"{w.name} seed {seed} vs regular: {k}", state_bf16=bf)


def test_sizes_beyond_the_static_workspace_are_rejected():
    torch = torch_mod()
    w = wl.MID                                   # needs ~200 MiB of workspace
    assert cfc.cfc_kloop_workspace_bytes(w.B, w.K, w.n_in, w.n_hid, w.math, wl.GRAD_GEMM) > 16 << 20
    lib = cfc.load_library()
    buf = torch.zeros(1024, device="cuda")
    p = buf.data_ptr()
    st = lib.cfc_kloop_forward_backward_static(p, p, p, p, p, p, 0, w.B, w.K, w.n_in, w.n_hid,
                                               w.math, None, None, p, p, p, p, p, None, None, None)
    assert st == -8 and "CFC_STATIC_WORKSPACE_BYTES" in cfc.cfc_status_string(st)
    torch.cuda.synchronize()
    assert torch.count_nonzero(buf).item() == 0  # nothing was launched
