"""Pins of the GRN-heads oracle against facts other than itself: central finite
differences of a loss on the probabilities, printed values of the normal CDF
(GELU(z) = z Phi(z)), the closed form with a zero first layer, the role of
lambda and of grad_h_carry, sample independence and the batch sum."""

import math

import numpy as np
import pytest

from oracle import grn_oracle as go

HD, M, J, B, K = 3, 2, 2, 2, 3


def _case(seed=0, Hd=HD, M_=M, J_=J, B_=B, K_=K):
    rng = np.random.default_rng(seed)
    N = go.grn_param_length(Hd, M_, J_)
    return dict(h=rng.standard_normal((B_ * K_, Hd)), params=rng.uniform(-0.8, 0.8, N),
                c=rng.standard_normal((B_ * K_, J_)), lam=rng.uniform(0.5, 1.5, J_),
                carry=rng.standard_normal((B_ * K_, Hd)))


def _loss(h, params, c, Hd=HD, M_=M, J_=J, horizon=None):
    p = go.grn_forward(h, params, Hd, M_, J_)["p"]
    if horizon is not None:
        return float(np.sum(c[:, horizon] * p[:, horizon]))
    return float(np.sum(c * p))


def test_param_length_matches_the_pages_count():
    # 12,675 parameters per horizon at HIDDEN = 128, HEAD_MID = 64; 63,375 for 5 horizons
    assert go.grn_param_length(128, 64, 1) == 12675
    assert go.grn_param_length(128, 64, 5) == 63375


def test_gelu_against_printed_normal_cdf():
    # Phi(1) = 0.841344746..., Phi(2) = 0.977249868..., Phi(-1) = 0.158655253...
    z = np.array([1.0, 2.0, -1.0, 0.0])
    phi = np.array([0.8413447460685429, 0.9772498680518208, 0.15865525393145707, 0.5])
    np.testing.assert_allclose(go.gelu(z), z * phi, rtol=1e-15, atol=1e-16)
    # the derivative against central differences, and its value 1/2 at 0
    zz = np.linspace(-4, 4, 33)
    e = 1e-6
    np.testing.assert_allclose(go.gelu_grad(zz), (go.gelu(zz + e) - go.gelu(zz - e)) / (2 * e), rtol=1e-8,
                               atol=1e-9)
    assert go.gelu_grad(np.array([0.0]))[0] == 0.5


def test_parameter_gradient_matches_central_differences():
    c = _case()
    g = go.grn_backward(c["h"], c["params"], c["c"], c["lam"], B, K, HD, M, J)
    num = np.zeros_like(c["params"])
    e = 1e-6
    for n in range(c["params"].size):
        pp, pm = c["params"].copy(), c["params"].copy()
        pp[n] += e
        pm[n] -= e
        num[n] = (_loss(c["h"], pp, c["c"]) - _loss(c["h"], pm, c["c"])) / (2 * e)
    np.testing.assert_allclose(g["grad_params"], num, rtol=1e-7, atol=1e-9)


@pytest.mark.parametrize("horizon", [0, 1])
def test_trunk_gradient_per_horizon_is_lambda_scaled(horizon):
    """grad_h - carry = sum_j lambda_j dL_j/dh, checked one horizon at a time."""
    c = _case(seed=1)
    lam = np.zeros(J)
    lam[horizon] = 1.7
    g = go.grn_backward(c["h"], c["params"], c["c"], lam, B, K, HD, M, J, grad_h_carry=c["carry"])
    num = np.zeros_like(c["h"])
    e = 1e-6
    for idx in np.ndindex(c["h"].shape):
        hp, hm = c["h"].copy(), c["h"].copy()
        hp[idx] += e
        hm[idx] -= e
        num[idx] = (_loss(hp, c["params"], c["c"], horizon=horizon)
                    - _loss(hm, c["params"], c["c"], horizon=horizon)) / (2 * e)
    np.testing.assert_allclose(g["grad_h"] - c["carry"], 1.7 * num, rtol=1e-7, atol=1e-9)


def test_lambda_zero_returns_the_carry_and_leaves_parameter_gradients():
    c = _case(seed=2)
    g0 = go.grn_backward(c["h"], c["params"], c["c"], np.zeros(J), B, K, HD, M, J, grad_h_carry=c["carry"])
    g1 = go.grn_backward(c["h"], c["params"], c["c"], c["lam"], B, K, HD, M, J, grad_h_carry=c["carry"])
    assert np.array_equal(g0["grad_h"], c["carry"])
    assert np.array_equal(g0["grad_params"], g1["grad_params"])


def test_zero_first_layer_closed_form():
    """W1 = b1 = 0: z1 = a1 = 0, z2 = b2, so every row's p is
    sigmoid(w_skip.h + b_skip + sigmoid(w_gate.b2 + b_gate)(w_main.b2 + b_main))."""
    c = _case(seed=3)
    P = go.unpack_grn(c["params"].copy(), HD, M, J)
    P["W1"][:] = 0.0
    P["b1"][:] = 0.0
    params = go.pack_grn(P, HD, M, J)
    f = go.grn_forward(c["h"], params, HD, M, J)
    for r in range(B * K):
        for j in range(J):
            gate = sum(P["w_gate"][j, m] * P["b2"][j, m] for m in range(M)) + P["b_gate"][j]
            main = sum(P["w_main"][j, m] * P["b2"][j, m] for m in range(M)) + P["b_main"][j]
            skip = sum(P["w_skip"][j, i] * c["h"][r, i] for i in range(HD)) + P["b_skip"][j]
            logit = skip + main / (1.0 + math.exp(-gate))
            assert abs(f["p"][r, j] - 1.0 / (1.0 + math.exp(-logit))) < 1e-15
            assert np.all(f["z1"][r, j] == 0.0) and np.all(f["a1"][r, j] == 0.0)


def test_samples_are_independent_and_rows_sum_to_the_batch_gradient():
    c = _case(seed=4, B_=3, K_=2)
    g = go.grn_backward(c["h"], c["params"], c["c"], c["lam"], 3, 2, HD, M, J)
    np.testing.assert_allclose(g["per_sample"].sum(0), g["grad_params"], rtol=1e-15)
    for b in range(3):
        rows = slice(2 * b, 2 * b + 2)
        one = go.grn_backward(c["h"][rows], c["params"], c["c"][rows], c["lam"], 1, 2, HD, M, J)
        np.testing.assert_allclose(one["per_sample"][0], g["per_sample"][b], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(one["grad_h"], g["grad_h"][rows], rtol=1e-12, atol=1e-15)


def test_pack_unpack_round_trip_and_segment_order():
    N = go.grn_param_length(HD, M, J)
    v = np.arange(N, dtype=np.float64)
    P = go.unpack_grn(v, HD, M, J)
    assert list(P) == list(go.GRN_SEGMENTS)
    assert P["W1"].shape == (J, M, HD) and P["W1"][0, 0, 0] == 0.0
    assert P["b_skip"][-1] == N - 1
    assert np.array_equal(go.pack_grn(P, HD, M, J), v)
