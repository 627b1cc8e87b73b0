"""Failure detection without a GPU fault: a bounded wait that runs out is
reported through the device error word, the word clears, and the context
keeps computing correct results afterwards."""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import workloads as wl

from gpu_common import PARITY_BIAS, CfcRun, assert_close, require_gpu, torch_mod

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_the_context_survives():
    require_gpu()
    torch = torch_mod()
    assert cfc.cfc_device_error(clear=True) == 0
    cfc.cfc_selftest_timeout(1000)
    torch.cuda.synchronize()
    assert cfc.cfc_device_error(clear=False) == 1       # reported
    assert cfc.cfc_device_error(clear=True) == 1        # read and cleared
    assert cfc.cfc_device_error() == 0
    # the same context still runs a step correctly
    w = wl.TINY
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r = CfcRun(w, inp)
    r.forward()
    r.backward()
    got = r.results()                                   # asserts the error word stays 0
    ref = oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"], y=inp["y"])
    for k in ("h_seq", "grad_W_in", "grad_W_rec", "grad_b", "grad_h0"):
        assert_close(got[k], ref[k], w.math, f"after timeout: {k}")
