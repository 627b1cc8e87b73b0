"""Pins of the tau-cell oracle against facts other than itself: central finite
differences of the loss, the closed form of the recurrence with zero
weights, the plain tanh RNN it reduces to when every tau is below the clamp,
the no-op limit of a huge tau, sample independence and the batch sum."""

import numpy as np
import pytest

from oracle import tau_oracle as to


def _case(B=2, K=3, n_in=3, H=4, seed=0, tau=None, dt=None):
    rng = np.random.default_rng(seed)
    c = dict(x=rng.standard_normal((B, K, n_in)), h0=rng.standard_normal((B, H)),
             W_in=rng.uniform(-0.6, 0.6, (H, n_in)), W_rec=rng.uniform(-0.5, 0.5, (H, H)),
             b=rng.uniform(-0.3, 0.3, H),
             tau=rng.uniform(0.5, 2.0, H) if tau is None else np.asarray(tau, dtype=np.float64),
             dt=rng.uniform(0.5, 1.5, B) if dt is None else np.asarray(dt, dtype=np.float64))
    c["y"] = rng.standard_normal((B, H))
    c["gseq"] = rng.standard_normal((B, K, H))
    return c


def _loss(c, **over):
    p = {**c, **over}
    f = to.tau_forward(p["x"], p["h0"], p["W_in"], p["W_rec"], p["b"], p["tau"], p["dt"])
    hs = f["h_seq"]
    return 0.5 * np.sum((hs[:, -1] - p["y"]) ** 2) + np.sum(p["gseq"] * hs)


@pytest.mark.parametrize("name", ["W_in", "W_rec", "b", "tau", "h0", "x"])
def test_gradients_match_central_differences(name):
    c = _case(tau=[0.7, 1.3, 1e-7, 2.0])         # one tau below the clamp: zero gradient
    g = to.tau_backward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"],
                        grad_h_seq=c["gseq"], y=c["y"])
    key = {"W_in": "grad_W_in", "W_rec": "grad_W_rec", "b": "grad_b", "tau": "grad_tau",
           "h0": "grad_h0", "x": "grad_x"}[name]
    base = c[name]
    num = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        eps = 1e-9 if (name == "tau" and base[idx] < to.TAU_EPS) else 1e-6
        p, m = base.copy(), base.copy()
        p[idx] += eps
        m[idx] -= eps
        num[idx] = (_loss(c, **{name: p}) - _loss(c, **{name: m})) / (2 * eps)
    np.testing.assert_allclose(g[key], num, rtol=1e-6, atol=1e-8)
    if name == "tau":
        assert g["grad_tau"][2] == 0.0


def test_clamped_tau_gets_no_gradient_while_its_decay_is_live():
    """A tau below the 1e-6 clamp enters the forward only as max(tau, 1e-6), so
    the loss is flat in it and its gradient is exactly 0 ("grad_tau only
    where tau > eps").  With a step dt of a few 1e-7 the clamped unit's decay
    exp(-dt / 1e-6) stays near 0.8 instead of underflowing, so a gradient
    formula that ignored the clamp would give a non-zero value here."""
    c = _case(tau=[0.7, 1.3, 5e-7, 2.0], dt=[2e-7, 3e-7])
    g = to.tau_backward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"],
                        grad_h_seq=c["gseq"], y=c["y"])
    num = np.zeros(4)
    for i in range(4):
        # the live units' gradients are ~1e-6 (dt / tau^2 scale): a wide step
        # keeps the difference quotient above the loss's rounding noise
        eps = 1e-9 if c["tau"][i] < to.TAU_EPS else 1e-3
        p, m = c["tau"].copy(), c["tau"].copy()
        p[i] += eps
        m[i] -= eps
        num[i] = (_loss(c, tau=p) - _loss(c, tau=m)) / (2 * eps)
    assert g["grad_tau"][2] == 0.0 and num[2] == 0.0
    np.testing.assert_allclose(g["grad_tau"], num, rtol=1e-4, atol=1e-12)
    assert np.all(np.abs(g["grad_tau"][[0, 1, 3]]) > 1e-9)      # the live units do move


def test_clamp_value_in_the_closed_form():
    """W = 0 with step sizes of a few 1e-7, so that the decay of units with
    tau near the clamp is neither 0 nor 1: h_K = s + decay^K (h0 - s) with
    decay = exp(-dt / max(tau, 1e-6)), the pages' constant written out here.
    Units below, at, just above and well above 1e-6; those above it get a
    non-zero tau gradient, the others exactly zero."""
    tau = np.array([5e-7, 1e-6, 3e-6, 1e-5, 1.0])
    dt = np.array([2e-7, 3e-7])
    c = _case(B=2, K=4, n_in=2, H=5, seed=13, tau=tau, dt=dt)
    c["W_in"][:] = 0.0
    c["W_rec"][:] = 0.0
    hs = to.tau_forward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"])["h_seq"]
    s = np.tanh(c["b"])[None, :]
    d = np.exp(-dt[:, None] / np.maximum(tau, 1e-6)[None, :])
    for k in range(4):
        np.testing.assert_allclose(hs[:, k], s + d ** (k + 1) * (c["h0"] - s), rtol=1e-13, atol=1e-14)
    g = to.tau_backward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"], y=c["y"])
    assert g["grad_tau"][0] == 0.0 and g["grad_tau"][1] == 0.0
    assert np.all(g["grad_tau"][2:] != 0.0)


def test_zero_weights_closed_form():
    """W_in = W_rec = 0: s = tanh(b) every step, so h_K = s + decay^K (h0 - s)."""
    c = _case(B=3, K=7, n_in=2, H=5, seed=3)
    c["W_in"][:] = 0.0
    c["W_rec"][:] = 0.0
    hs = to.tau_forward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"])["h_seq"]
    s = np.tanh(c["b"])[None, :]
    d = np.exp(-c["dt"][:, None] / c["tau"][None, :])
    for k in range(7):
        np.testing.assert_allclose(hs[:, k], s + d ** (k + 1) * (c["h0"] - s), rtol=1e-13, atol=1e-14)


def test_tau_below_clamp_is_the_tanh_rnn():
    """Every tau below 1e-6: decay = exp(-dt / 1e-6) underflows to 0, the cell is
    h' = tanh(W_in x + W_rec h + b), and no gradient reaches tau."""
    c = _case(B=2, K=4, n_in=3, H=3, seed=5, tau=[1e-8, 5e-7, 1e-9], dt=[1.0, 0.5])
    hs = to.tau_forward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"])["h_seq"]
    h = c["h0"]
    for k in range(4):
        h = np.tanh(np.einsum("ij,bj->bi", c["W_in"], c["x"][:, k]) + np.einsum("ij,bj->bi", c["W_rec"], h)
                    + c["b"])
        np.testing.assert_allclose(hs[:, k], h, rtol=1e-14, atol=1e-15)
    g = to.tau_backward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"], y=c["y"])
    assert np.all(g["grad_tau"] == 0.0)


def test_huge_tau_keeps_the_state():
    c = _case(B=2, K=5, seed=7, tau=[1e12] * 4)
    hs = to.tau_forward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"])["h_seq"]
    np.testing.assert_allclose(hs[:, -1], c["h0"], atol=1e-10)


def test_samples_are_independent_and_rows_sum_to_the_batch_gradient():
    c = _case(B=3, K=4, n_in=2, H=3, seed=11)
    full = to.tau_backward(c["x"], c["h0"], c["W_in"], c["W_rec"], c["b"], c["tau"], c["dt"],
                           grad_h_seq=c["gseq"], y=c["y"])
    for bi in range(3):
        one = to.tau_backward(c["x"][bi:bi + 1], c["h0"][bi:bi + 1], c["W_in"], c["W_rec"], c["b"], c["tau"],
                              c["dt"][bi:bi + 1], grad_h_seq=c["gseq"][bi:bi + 1], y=c["y"][bi:bi + 1])
        # equal up to the BLAS summation order of a different batch size
        np.testing.assert_allclose(one["per_sample"][0], full["per_sample"][bi], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(one["h_seq"][0], full["h_seq"][bi], rtol=1e-12, atol=1e-15)
    gWi, gWr, gb, gtau = to.unpack_tau_per_sample(full["per_sample"], 2, 3)
    np.testing.assert_allclose(gWi.sum(0), full["grad_W_in"], rtol=1e-14)
    np.testing.assert_allclose(gWr.sum(0), full["grad_W_rec"], rtol=1e-14)
    np.testing.assert_allclose(gb.sum(0), full["grad_b"], rtol=1e-14)
    np.testing.assert_allclose(gtau.sum(0), full["grad_tau"], rtol=1e-14)
    assert full["per_sample"].shape[1] == to.tau_per_sample_length(2, 3)
