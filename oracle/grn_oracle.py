"""CPU oracle for the multi-horizon GRN heads evaluated on every K position of
the trunk state, forward and backward.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the CPU
baseline leg of the benchmark may import or run this module.  It shares no
code with the CUDA path and never takes an input or an expected value from it.
Plain numpy, float64.

Source: the ml-alpha commit history page (crates/ml-alpha/src), commit
b6dfd89903 "wire TFT GRN heads into PerceptionTrainer (Phase 1.7)", gives the
forward composition per horizon j of the trunk state h (length Hd):

    z1   = W1[j] h + b1[j]                       [M]   (W1: HIDDEN -> HEAD_MID)
    a1   = GELU(z1)
    z2   = W2[j] a1 + b2[j]                      [M]   (W2: HEAD_MID -> HEAD_MID)
    gate = w_gate[j] . z2 + b_gate[j]                  (the "gate_lin" head)
    main = w_main[j] . z2 + b_main[j]
    skip = w_skip[j] . h  + b_skip[j]                  (W_skip: HIDDEN -> 1)
    logit = skip + sigmoid(gate) * main
    p     = sigmoid(logit)

with ten parameter tensors per horizon, saved intermediates z1, a1, z2 and
gate, main per K position, and the heads run at every K position of the K
loop.  "K-loop Parallelization Implementation Plan", Commit 2 / Task 11 gives
the backward's contract: inputs probs, grad_probs (dL/dp), the saved
intermediates, h, grad_h_carry and a per-horizon lambda that scales only the
trunk gradient; outputs the ten parameter gradients accumulated (+=) into
per-sample scratch rows over the K positions of the loop (k from K-1 down to
0) and grad_h (overwrite).  The pages leave the chain-rule body to a kernel
they do not print; it is the derivative of the forward above:

    dlogit = grad_p * p (1 - p);   dskip = dlogit
    dmain  = dlogit * sigmoid(gate);  dgate = dlogit * main * sigmoid'(gate)
    dz2    = dmain * w_main + dgate * w_gate
    dz1    = (W2^T dz2) * GELU'(z1)
    grad_h = grad_h_carry + sum_j lambda_j (W1[j]^T dz1_j + dskip_j w_skip[j])

Readings: GELU is the exact form z * Phi(z) (the pages name GELU without a
variant); grad_h_carry is added to the heads' trunk gradient (the pages pass
it in and write grad_h whole); rows are r = b*K + k (sample-major, the layout
of the K loop's h_seq), so grad_h feeds the K loop's per-step upstream
gradient.  The packed parameter (and gradient) vector holds the ten tensors
in the pages' order, each horizon-major:
[W1 (J,M,Hd) | b1 (J,M) | W2 (J,M,M) | b2 (J,M) | w_gate (J,M) | b_gate (J) |
 w_main (J,M) | b_main (J) | w_skip (J,Hd) | b_skip (J)].
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

GRN_SEGMENTS = ("W1", "b1", "W2", "b2", "w_gate", "b_gate", "w_main", "b_main", "w_skip", "b_skip")


def grn_shapes(Hd: int, M: int, J: int) -> dict:
    return {"W1": (J, M, Hd), "b1": (J, M), "W2": (J, M, M), "b2": (J, M), "w_gate": (J, M),
            "b_gate": (J,), "w_main": (J, M), "b_main": (J,), "w_skip": (J, Hd), "b_skip": (J,)}


def grn_param_length(Hd: int, M: int, J: int) -> int:
    """J (M Hd + M + M M + M + M + 1 + M + 1 + Hd + 1)."""
    return sum(int(np.prod(s)) for s in grn_shapes(Hd, M, J).values())


def unpack_grn(vec, Hd: int, M: int, J: int) -> dict:
    """Split a packed [..., N] vector into the ten tensors (views)."""
    vec = np.asarray(vec)
    lead = vec.shape[:-1]
    out, o = {}, 0
    for name, shp in grn_shapes(Hd, M, J).items():
        n = int(np.prod(shp))
        out[name] = vec[..., o:o + n].reshape(*lead, *shp)
        o += n
    return out


def pack_grn(tensors: dict, Hd: int, M: int, J: int) -> np.ndarray:
    parts = []
    for name, shp in grn_shapes(Hd, M, J).items():
        t = np.asarray(tensors[name], dtype=np.float64)
        lead = t.shape[:t.ndim - len(shp)]
        parts.append(t.reshape(*lead, -1))
    return np.concatenate(parts, axis=-1)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def gelu(z):
    """z * Phi(z), Phi the standard normal CDF."""
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def gelu_grad(z):
    """Phi(z) + z phi(z)."""
    return 0.5 * (1.0 + erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def grn_forward(h, params, Hd: int, M: int, J: int) -> dict:
    """h [R, Hd] -> z1, a1, z2 [R, J, M]; gate, main, skip, logit, p [R, J]."""
    h = np.asarray(h, dtype=np.float64)
    P = unpack_grn(np.asarray(params, dtype=np.float64), Hd, M, J)
    z1 = np.einsum("jmi,ri->rjm", P["W1"], h) + P["b1"][None]
    a1 = gelu(z1)
    z2 = np.einsum("jmn,rjn->rjm", P["W2"], a1) + P["b2"][None]
    gate = np.einsum("jm,rjm->rj", P["w_gate"], z2) + P["b_gate"][None]
    main = np.einsum("jm,rjm->rj", P["w_main"], z2) + P["b_main"][None]
    skip = h @ P["w_skip"].T + P["b_skip"][None]
    logit = skip + sigmoid(gate) * main
    return dict(z1=z1, a1=a1, z2=z2, gate=gate, main=main, skip=skip, logit=logit, p=sigmoid(logit))


def grn_backward(h, params, grad_probs, lam, B: int, K: int, Hd: int, M: int, J: int,
                 grad_h_carry=None) -> dict:
    """Rows r = b*K + k.  Returns grad_h [R, Hd], per_sample [B, N] (each
    sample's parameter gradient summed over k = K-1 .. 0), grad_params [N]
    (the sum over the batch) and the forward's intermediates."""
    h = np.asarray(h, dtype=np.float64)
    R = h.shape[0]
    assert R == B * K
    P = unpack_grn(np.asarray(params, dtype=np.float64), Hd, M, J)
    f = grn_forward(h, params, Hd, M, J)
    gp = np.asarray(grad_probs, dtype=np.float64)
    lam = np.asarray(lam, dtype=np.float64)
    p = f["p"]
    dlogit = gp * p * (1.0 - p)
    sg = sigmoid(f["gate"])
    dskip = dlogit
    dmain = dlogit * sg
    dgate = dlogit * f["main"] * sg * (1.0 - sg)
    dz2 = dmain[:, :, None] * P["w_main"][None] + dgate[:, :, None] * P["w_gate"][None]
    da1 = np.einsum("jmn,rjm->rjn", P["W2"], dz2)
    dz1 = da1 * gelu_grad(f["z1"])
    trunk = np.einsum("jmi,rjm->rji", P["W1"], dz1) + dskip[:, :, None] * P["w_skip"][None]
    grad_h = np.einsum("j,rji->ri", lam, trunk)
    if grad_h_carry is not None:
        grad_h = grad_h + np.asarray(grad_h_carry, dtype=np.float64)

    # per-row parameter gradients, then summed per sample over k descending
    rows = {
        "W1": dz1[:, :, :, None] * h[:, None, None, :],
        "b1": dz1,
        "W2": dz2[:, :, :, None] * f["a1"][:, :, None, :],
        "b2": dz2,
        "w_gate": dgate[:, :, None] * f["z2"],
        "b_gate": dgate,
        "w_main": dmain[:, :, None] * f["z2"],
        "b_main": dmain,
        "w_skip": dskip[:, :, None] * h[:, None, :],
        "b_skip": dskip,
    }
    per_row = pack_grn(rows, Hd, M, J).reshape(B, K, -1)
    per_sample = np.zeros((B, per_row.shape[-1]))
    for k in range(K - 1, -1, -1):
        per_sample += per_row[:, k]
    return dict(grad_h=grad_h, per_sample=per_sample, grad_params=per_sample.sum(0),
                dz1=dz1, dz2=dz2, dgate=dgate, dmain=dmain, dskip=dskip, **f)
