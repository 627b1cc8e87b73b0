"""Pins of the CPU oracle's cell arithmetic against things other than itself:
hand-derived golden values, closed forms, a library RNN, finite differences
and structural invariants.  CPU only."""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import FP32, TF32, BF16
from recurrent_cell_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(B, K, n_in, H, seed=1, dt=None, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, K, n_in))
    h0 = rng.standard_normal((B, H))
    W_in = rng.uniform(-1, 1, (3, H, n_in)) * scale / math.sqrt(n_in)
    W_rec = rng.uniform(-1, 1, (3, H, H)) * scale / math.sqrt(H)
    b = rng.uniform(-0.3, 0.3, (3, H))
    if dt is None:
        dt = rng.uniform(0.5, 1.5, B)
    return x, h0, W_in, W_rec, b, dt


# ---------------------------------------------------------------- rounding

def test_bf16_rounding_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    a = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
        # exact ties: bf16 value + half an ulp
        (np.float32(1.0) + np.float32(2.0 ** -8)) * np.ones(1, np.float32),
        (np.float32(1.0) + np.float32(3 * 2.0 ** -8)) * np.ones(1, np.float32),
    ])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(a), ref)


def test_tf32_rounding_definition():
    one = 1.0
    cases = [
        (one + 2.0 ** -11, one + 2.0 ** -10),                  # tie -> away from zero
        (-(one + 2.0 ** -11), -(one + 2.0 ** -10)),
        (one + 2.0 ** -11 - 2.0 ** -23, one),                  # just below the tie
        (one + 3 * 2.0 ** -11, one + 2.0 ** -9),               # tie on an odd step, away
        (one + 2.0 ** -10, one + 2.0 ** -10),                  # representable
        (0.0, 0.0),
    ]
    for a, want in cases:
        assert oracle.round_tf32(np.array([a]))[0] == want, a
    rng = np.random.default_rng(4)
    a = rng.standard_normal(10000).astype(np.float32)
    r = oracle.round_tf32(a)
    bits = r.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0x1FFF == 0)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(a.astype(np.float64)))) - 10)
    assert np.all(np.abs(r - a) <= ulp / 2 + 1e-30)


# ---------------------------------------------------------------- golden

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([f.strip() for f in line.split(";")])
    return rows


def test_scalar_step_golden():
    L3, L2 = math.log(3.0), math.log(2.0)
    for name, dt, wf, seed, h1, dAf, dAg, dAh in _read_golden("cfc_scalar_step.txt"):
        dt = float(dt)
        W_in_f = {"L3": L3, "L3/2": L3 / 2}[wf]
        W_in = np.array([W_in_f, L2, L3]).reshape(3, 1, 1)
        W_rec = np.array([0.5, -0.25, 2.0]).reshape(3, 1, 1)
        b = np.zeros((3, 1))
        x = np.ones((1, 1, 1))
        h0 = np.zeros((1, 1))
        kw = {}
        if seed.startswith("grad_h_last="):
            kw["grad_h_last"] = np.full((1, 1), float(seed.split("=")[1]))
        else:
            kw["y"] = np.full((1, 1), float(seed.split("=")[1]))
        fw = oracle.forward(x, h0, W_in, W_rec, b, dt)
        assert fw["h_seq"][0, 0, 0] == pytest.approx(float(h1), abs=1e-14), name
        bw = oracle.backward(x, h0, W_in, W_rec, b, dt, **kw)
        dA = np.array([float(dAf), float(dAg), float(dAh)])
        np.testing.assert_allclose(bw["grad_b"][:, 0], dA, atol=1e-14, err_msg=name)
        np.testing.assert_allclose(bw["grad_W_in"][:, 0, 0], dA, atol=1e-14, err_msg=name)
        np.testing.assert_allclose(bw["grad_W_rec"][:, 0, 0], 0.0, atol=1e-14, err_msg=name)
        gh0 = 0.5 * dA[0] - 0.25 * dA[1] + 2.0 * dA[2]
        gx = W_in_f * dA[0] + L2 * dA[1] + L3 * dA[2]
        assert bw["grad_h0"][0, 0] == pytest.approx(gh0, abs=1e-14), name
        assert bw["grad_x"][0, 0, 0] == pytest.approx(gx, abs=1e-14), name


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("K", [1, 3])
def test_zero_weights_closed_form(K):
    """W = 0, b = 0: every head is 0, gate = 1/2, h_k = 0 for k >= 1.  With the
    loss 0.5||h_K - y||^2 only step K-1 receives a gradient, delta = -y."""
    B, n_in, H = 3, 4, 5
    rng = np.random.default_rng(7)
    x = rng.standard_normal((B, K, n_in))
    h0 = rng.standard_normal((B, H))
    y = rng.standard_normal((B, H))
    W_in = np.zeros((3, H, n_in))
    W_rec = np.zeros((3, H, H))
    b = np.zeros((3, H))
    dt = 0.7
    fw = oracle.forward(x, h0, W_in, W_rec, b, dt)
    assert np.all(fw["h_seq"] == 0.0)
    assert np.all(fw["gate"] == 0.5)
    bw = oracle.backward(x, h0, W_in, W_rec, b, dt, y=y)
    gWi, gWr, gb = oracle.unpack_per_sample(bw["per_sample"], n_in, H)
    np.testing.assert_array_equal(gb[:, 0], 0.0)
    np.testing.assert_allclose(gb[:, 1], -0.5 * y, rtol=0, atol=1e-15)
    np.testing.assert_allclose(gb[:, 2], -0.5 * y, rtol=0, atol=1e-15)
    for c in (1, 2):
        np.testing.assert_allclose(gWi[:, c], np.einsum("bi,bj->bij", -0.5 * y, x[:, K - 1]),
                                   atol=1e-15)
        want_rec = np.einsum("bi,bj->bij", -0.5 * y, h0) if K == 1 else 0.0
        np.testing.assert_allclose(gWr[:, c], want_rec, atol=1e-15)
    np.testing.assert_array_equal(gWi[:, 0], 0.0)
    np.testing.assert_array_equal(gWr[:, 0], 0.0)
    np.testing.assert_array_equal(bw["grad_h0"], 0.0)
    np.testing.assert_array_equal(bw["grad_x"], 0.0)


def test_dt_zero_freezes_gate():
    """dt = 0: gate = sigmoid(0) = 1/2 whatever f is, so every f-head gradient is 0."""
    x, h0, W_in, W_rec, b, _ = _rand_problem(2, 4, 3, 5, seed=11)
    y = np.random.default_rng(12).standard_normal((2, 5))
    fw = oracle.forward(x, h0, W_in, W_rec, b, 0.0)
    assert np.all(fw["gate"] == 0.5)
    bw = oracle.backward(x, h0, W_in, W_rec, b, 0.0, y=y)
    assert np.all(bw["grad_W_in"][0] == 0.0)
    assert np.all(bw["grad_W_rec"][0] == 0.0)
    assert np.all(bw["grad_b"][0] == 0.0)
    assert np.any(bw["grad_W_in"][1] != 0.0)


@pytest.mark.parametrize("bf, head", [(10.0, 2), (-10.0, 1)])
def test_saturated_gate_is_elman_rnn(bf, head):
    """W_f = 0, b_f = +10, dt = 100: gate = 1/(1+e^1000) = 0 exactly, so
    h' = tanh(W_in[h~] x + W_rec[h~] h + b[h~]) -- an Elman tanh RNN.  b_f = -10
    gives gate = 1 and h' = tanh(W_in[g] x + ...).  Forward and gradients are
    compared with torch.nn.RNN in float64 and autograd."""
    torch = pytest.importorskip("torch")
    B, K, n_in, H = 3, 5, 4, 6
    x, h0, W_in, W_rec, b, _ = _rand_problem(B, K, n_in, H, seed=21)
    W_in[0] = 0.0
    W_rec[0] = 0.0
    b[0] = bf
    y = np.random.default_rng(22).standard_normal((B, H))
    G = np.random.default_rng(23).standard_normal((B, K, H))
    fw = oracle.forward(x, h0, W_in, W_rec, b, 100.0)
    bw = oracle.backward(x, h0, W_in, W_rec, b, 100.0, y=y, grad_h_seq=G)

    rnn = torch.nn.RNN(n_in, H, nonlinearity="tanh", batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        rnn.weight_ih_l0.copy_(torch.from_numpy(W_in[head]))
        rnn.weight_hh_l0.copy_(torch.from_numpy(W_rec[head]))
        rnn.bias_ih_l0.copy_(torch.from_numpy(b[head]))
        rnn.bias_hh_l0.zero_()
    xt = torch.from_numpy(x).requires_grad_(True)
    h0t = torch.from_numpy(h0)[None].clone().requires_grad_(True)
    out, _ = rnn(xt, h0t)
    loss = 0.5 * ((out[:, -1] - torch.from_numpy(y)) ** 2).sum() + (out * torch.from_numpy(G)).sum()
    loss.backward()
    np.testing.assert_allclose(fw["h_seq"], out.detach().numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(bw["grad_W_in"][head], rnn.weight_ih_l0.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(bw["grad_W_rec"][head], rnn.weight_hh_l0.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(bw["grad_b"][head], rnn.bias_ih_l0.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(bw["grad_h0"], h0t.grad[0].numpy(), atol=1e-12)
    np.testing.assert_allclose(bw["grad_x"], xt.grad.numpy(), atol=1e-12)
    other = 1 if head == 2 else 2
    for c in (0, other):
        assert np.all(bw["grad_W_in"][c] == 0.0)
        assert np.all(bw["grad_b"][c] == 0.0)


# ---------------------------------------------------------------- finite differences

def _loss(x, h0, W_in, W_rec, b, dt, y, G, Gl):
    hs = oracle.forward(x, h0, W_in, W_rec, b, dt)["h_seq"]
    return (0.5 * np.sum((hs[:, -1] - y) ** 2) + np.sum(hs * G) + np.sum(hs[:, -1] * Gl))


def test_finite_differences_every_element_tiny():
    """Central differences (float64, eps 1e-6) on EVERY element of W_in, W_rec,
    b, h0 and x of the tiny workload (B=4, K=8, n_in=16, n_hid=32), with a
    loss that exercises all three upstream seeds (y, grad_h_seq, grad_h_last)."""
    w = wl.TINY
    inp = wl.make_inputs(w)
    rng = np.random.default_rng(5)
    x = inp["x"].astype(np.float64)
    h0 = inp["h0"].astype(np.float64)
    W_in = inp["W_in"].astype(np.float64)
    W_rec = inp["W_rec"].astype(np.float64)
    b = rng.uniform(-0.2, 0.2, (3, w.n_hid))
    dt = rng.uniform(0.5, 1.5, w.B)
    y = inp["y"].astype(np.float64)
    G = 0.1 * rng.standard_normal((w.B, w.K, w.n_hid))
    Gl = 0.3 * rng.standard_normal((w.B, w.n_hid))
    bw = oracle.backward(x, h0, W_in, W_rec, b, dt, y=y, grad_h_seq=G, grad_h_last=Gl)
    args = dict(x=x, h0=h0, W_in=W_in, W_rec=W_rec, b=b)
    grads = dict(x=bw["grad_x"], h0=bw["grad_h0"], W_in=bw["grad_W_in"],
                 W_rec=bw["grad_W_rec"], b=bw["grad_b"])
    eps = 1e-6
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + eps
            lp = _loss(dt=dt, y=y, G=G, Gl=Gl, **args)
            flat[idx] = old - eps
            lm = _loss(dt=dt, y=y, G=G, Gl=Gl, **args)
            flat[idx] = old
            fd.reshape(-1)[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


# ---------------------------------------------------------------- invariants

def test_batch_rows_independent_and_permutation_equivariant():
    x, h0, W_in, W_rec, b, dt = _rand_problem(5, 6, 3, 4, seed=31)
    y = np.random.default_rng(32).standard_normal((5, 4))
    full = oracle.backward(x, h0, W_in, W_rec, b, dt, y=y)
    for i in range(5):                      # B = 1 equals the row of the batch
        one = oracle.backward(x[i:i + 1], h0[i:i + 1], W_in, W_rec, b, dt[i:i + 1], y=y[i:i + 1])
        np.testing.assert_allclose(one["h_seq"][0], full["h_seq"][i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(one["per_sample"][0], full["per_sample"][i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(one["grad_h0"][0], full["grad_h0"][i], rtol=0, atol=1e-14)
    perm = np.array([3, 0, 4, 1, 2])
    pb = oracle.backward(x[perm], h0[perm], W_in, W_rec, b, dt[perm], y=y[perm])
    np.testing.assert_allclose(pb["h_seq"], full["h_seq"][perm], rtol=0, atol=1e-14)
    np.testing.assert_allclose(pb["grad_x"], full["grad_x"][perm], rtol=0, atol=1e-14)
    np.testing.assert_allclose(pb["per_sample"], full["per_sample"][perm], rtol=0, atol=1e-13)
    np.testing.assert_allclose(pb["grad_W_rec"], full["grad_W_rec"], rtol=1e-13, atol=1e-13)


def test_reduced_gradient_is_sum_of_per_sample():
    x, h0, W_in, W_rec, b, dt = _rand_problem(6, 3, 5, 4, seed=41)
    bw = oracle.backward(x, h0, W_in, W_rec, b, dt, y=np.ones((6, 4)))
    gWi, gWr, gb = oracle.unpack_per_sample(bw["per_sample"].sum(0), 5, 4)
    np.testing.assert_allclose(gWi, bw["grad_W_in"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(gWr, bw["grad_W_rec"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(gb, bw["grad_b"], rtol=1e-14, atol=1e-15)
    assert bw["per_sample"].shape[1] == oracle.per_sample_length(5, 4) == 3 * (5 + 4 + 1) * 4


@pytest.mark.parametrize("mode, rnd", [(BF16, oracle.round_bf16), (TF32, oracle.round_tf32)])
def test_mode_rounding_points_single_step(mode, rnd):
    """At K = 1 with operands already representable in the mode's type, the
    reduced-precision modes differ from FP32 only at their stated rounding
    points: the stored state (bf16 only) and dA fed to the gradients."""
    B, n_in, H = 4, 3, 5
    x, h0, W_in, W_rec, b, dt = _rand_problem(B, 1, n_in, H, seed=51)
    x, h0, W_in, W_rec = (rnd(a) for a in (x, h0, W_in, W_rec))
    gl = np.random.default_rng(52).standard_normal((B, H))
    ref = oracle.backward(x, h0, W_in, W_rec, b, dt, FP32, grad_h_last=gl)
    got = oracle.backward(x, h0, W_in, W_rec, b, dt, mode, grad_h_last=gl)
    want_h = oracle.round_bf16(ref["h_seq"]) if mode == BF16 else ref["h_seq"]
    np.testing.assert_array_equal(got["h_seq"], want_h)
    # per-sample grad_b row == dA of that sample, rounded at the operand point
    _, _, gb_ref = oracle.unpack_per_sample(ref["per_sample"], n_in, H)
    gWi, gWr, gb = oracle.unpack_per_sample(got["per_sample"], n_in, H)
    np.testing.assert_array_equal(gb, rnd(gb_ref))
    np.testing.assert_allclose(gWi, np.einsum("bci,bj->bcij", gb, x[:, 0]), rtol=1e-15, atol=0)
    np.testing.assert_allclose(gWr, np.einsum("bci,bj->bcij", gb, h0), rtol=1e-15, atol=0)


@pytest.mark.parametrize("mode, rnd", [(BF16, oracle.round_bf16), (TF32, oracle.round_tf32)])
def test_mode_rounds_every_contraction_operand(mode, rnd):
    """Unrounded float64 inputs over K = 3 steps.  Forward: each step of a
    reduced-precision mode is an FP32 step on operands rounded to the mode's
    type (x_k, h_k, W_in, W_rec), and only BF16 rounds the carried state (h0
    arrives bf16 in that mode).  Backward: dA is mode-valued, and grad_x,
    grad_h0 and the weight gradients are its contractions with the rounded
    W_in, W_rec, x_k and h_k."""
    B, K, n_in, H = 3, 3, 4, 5
    x, h0, W_in, W_rec, b, dt = _rand_problem(B, K, n_in, H, seed=61)
    got = oracle.backward(x, h0, W_in, W_rec, b, dt, mode, y=np.ones((B, H)))
    h = rnd(h0) if mode == BF16 else h0
    hs = [h]
    for k in range(K):
        h_next = oracle.cell_forward(rnd(x[:, k]), rnd(h), rnd(W_in), rnd(W_rec), b, dt, FP32)[0]
        if mode == BF16:
            h_next = rnd(h_next)
        np.testing.assert_array_equal(got["h_seq"][:, k], h_next)
        h = h_next
        hs.append(h)
    dA = got["dA"].reshape(B, K, 3 * H)
    np.testing.assert_array_equal(rnd(dA), dA)
    assert np.any(dA != 0.0)
    for k in range(K):
        np.testing.assert_allclose(got["grad_x"][:, k], dA[:, k] @ rnd(W_in).reshape(3 * H, n_in),
                                   rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(got["grad_h0"], dA[:, 0] @ rnd(W_rec).reshape(3 * H, H), rtol=1e-14, atol=1e-15)
    gWi = np.einsum("bkc,bkj->cj", dA, rnd(x)).reshape(3, H, n_in)
    gWr = np.einsum("bkc,bkj->cj", dA, rnd(np.stack(hs[:-1], axis=1))).reshape(3, H, H)
    np.testing.assert_allclose(got["grad_W_in"], gWi, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(got["grad_W_rec"], gWr, rtol=1e-13, atol=1e-15)
