"""The seeded input generator: the parity tests' nonzero bias leaves every
other input of a seed unchanged and gives each head its own values."""

import numpy as np

from recurrent_cell_gb300 import workloads as wl


def test_bias_drawn_last_and_distinct_per_head():
    for w in (wl.TINY, wl.MID.with_(B=16, K=4), wl.LARGE.with_(B=8, K=2)):
        plain = wl.make_inputs(w, seed=4)
        biased = wl.make_inputs(w, seed=4, bias_scale=0.5)
        for k in ("x", "h0", "W_in", "W_rec", "y", "dt"):
            np.testing.assert_array_equal(plain[k], biased[k], err_msg=k)
        assert not np.any(plain["b"])
        b = biased["b"]
        assert b.shape == (3, w.n_hid) and np.all(np.abs(b) <= 0.5)
        # f, g and h~ biases differ from one another at every unit
        assert np.all(b[0] != b[1]) and np.all(b[1] != b[2]) and np.all(b[0] != b[2])


def test_tau_bias_drawn_last():
    w = wl.TAU_TINY
    plain = wl.make_tau_inputs(w, seed=4)
    biased = wl.make_tau_inputs(w, seed=4, bias_scale=0.5)
    for k in ("x", "h0", "W_in", "W_rec", "tau", "y", "dt"):
        np.testing.assert_array_equal(plain[k], biased[k], err_msg=k)
    assert not np.any(plain["b"]) and np.all(biased["b"] != 0)
