"""CPU oracle for the single-head tau-cell K loop (forward and
backward-through-time), the second cell of the pages.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the CPU
baseline leg of the benchmark may import or run this module.  It shares no
code with the CUDA path and never takes an input or an expected value from it.
Plain numpy, float64.

Source: "K-loop Parallelization Implementation Plan", Task 2 (forward kernel
cfc_step_batched) and Task 3 (backward kernel cfc_step_backward_batched).
Per sample b, unit i, step k (state h_k, input x_k):

    pre_i   = b_i + sum_j W_in[i, j] x_k[j] + sum_j W_rec[i, j] h_k[j]
    s_i     = tanh(pre_i)
    decay_i = exp(-dt / max(tau_i, 1e-6))
    h_{k+1, i} = h_{k, i} * decay_i + (1 - decay_i) * s_i

and, given the gradient dh reaching h_{k+1},

    d_pre_i    = dh_i (1 - decay_i) (1 - s_i^2)
    gb_i      += d_pre_i,  gW_in[i, j] += d_pre_i x_k[j],  gW_rec[i, j] += d_pre_i h_k[j]
    gtau_i    += dh_i (h_{k, i} - s_i) decay_i dt / max(tau_i, 1e-6)^2   only where tau_i > 1e-6
    grad h_k   = W_rec^T d_pre + dh * decay
    grad x_k   = W_in^T d_pre

The pages take one scalar dt; here dt may also be one value per sample (the
same readings as the three-head cell: a [B] array, or [1] broadcast).  The
loss seeds are those of the three-head oracle: grad_h_seq per step,
grad_h_last, and h_K - y for the loss 0.5 ||h_K - y||^2.
"""

from __future__ import annotations

import numpy as np

TAU_EPS = 1e-6


def _dt_vector(dt, B: int) -> np.ndarray:
    dt = np.asarray(dt, dtype=np.float64).reshape(-1)
    return np.full(B, dt[0]) if dt.size == 1 else dt


def tau_per_sample_length(n_in: int, H: int) -> int:
    """Packed per-sample gradient length (n_in + H + 2) * H:
    [gW_in (i, j) | gW_rec (i, j) | gb (i) | gtau (i)]."""
    return (n_in + H + 2) * H


def tau_decay(tau, dt_b):
    """decay[b, i] = exp(-dt_b / max(tau_i, 1e-6))."""
    tau_eff = np.maximum(np.asarray(tau, dtype=np.float64), TAU_EPS)
    return np.exp(-np.asarray(dt_b, dtype=np.float64)[:, None] / tau_eff[None, :])


def tau_forward(x, h0, W_in, W_rec, b, tau, dt) -> dict:
    """h_seq[:, k] = h_{k+1}; s[:, k] = tanh(pre) of step k."""
    x = np.asarray(x, dtype=np.float64)
    B, K, _ = x.shape
    h = np.asarray(h0, dtype=np.float64).copy()
    H = h.shape[1]
    Wi = np.asarray(W_in, dtype=np.float64)
    Wr = np.asarray(W_rec, dtype=np.float64)
    bb = np.asarray(b, dtype=np.float64)
    d = tau_decay(tau, _dt_vector(dt, B))
    h_seq = np.empty((B, K, H))
    s_all = np.empty((B, K, H))
    for k in range(K):
        s = np.tanh(bb + x[:, k] @ Wi.T + h @ Wr.T)
        h = h * d + (1.0 - d) * s
        h_seq[:, k] = h
        s_all[:, k] = s
    return dict(h_seq=h_seq, s=s_all)


def tau_backward(x, h0, W_in, W_rec, b, tau, dt, grad_h_seq=None, grad_h_last=None, y=None) -> dict:
    """Gradients of the loss through the K loop: grad_W_in [H, n_in],
    grad_W_rec [H, H], grad_b [H], grad_tau [H] (summed over the batch),
    grad_h0 [B, H], grad_x [B, K, n_in], h_seq, and the packed per-sample
    rows per_sample [B, (n_in + H + 2) H]."""
    x = np.asarray(x, dtype=np.float64)
    B, K, n_in = x.shape
    h0 = np.asarray(h0, dtype=np.float64)
    H = h0.shape[1]
    Wi = np.asarray(W_in, dtype=np.float64)
    Wr = np.asarray(W_rec, dtype=np.float64)
    tau = np.asarray(tau, dtype=np.float64)
    dtv = _dt_vector(dt, B)
    d = tau_decay(tau, dtv)
    tau_eff = np.maximum(tau, TAU_EPS)
    live = tau > TAU_EPS
    fw = tau_forward(x, h0, W_in, W_rec, b, tau, dt)
    h_seq, s_all = fw["h_seq"], fw["s"]
    h_prev = np.concatenate([h0[:, None], h_seq[:, :-1]], axis=1)

    gWi = np.zeros((B, H, n_in))
    gWr = np.zeros((B, H, H))
    gb = np.zeros((B, H))
    gtau = np.zeros((B, H))
    grad_x = np.zeros((B, K, n_in))
    carry = np.zeros((B, H))
    for k in range(K - 1, -1, -1):
        dh = carry.copy()
        if grad_h_seq is not None:
            dh += np.asarray(grad_h_seq, dtype=np.float64)[:, k]
        if k == K - 1:
            if grad_h_last is not None:
                dh += np.asarray(grad_h_last, dtype=np.float64)
            if y is not None:
                dh += h_seq[:, K - 1] - np.asarray(y, dtype=np.float64)
        s, hp = s_all[:, k], h_prev[:, k]
        d_pre = dh * (1.0 - d) * (1.0 - s * s)
        gb += d_pre
        gWi += d_pre[:, :, None] * x[:, k][:, None, :]
        gWr += d_pre[:, :, None] * hp[:, None, :]
        gtau += np.where(live[None, :], dh * (hp - s) * d * dtv[:, None] / (tau_eff * tau_eff)[None, :], 0.0)
        grad_x[:, k] = d_pre @ Wi
        carry = d_pre @ Wr + dh * d
    per_sample = np.concatenate([gWi.reshape(B, -1), gWr.reshape(B, -1), gb, gtau], axis=1)
    return dict(grad_W_in=gWi.sum(0), grad_W_rec=gWr.sum(0), grad_b=gb.sum(0), grad_tau=gtau.sum(0),
                grad_h0=carry, grad_x=grad_x, h_seq=h_seq, per_sample=per_sample)


def unpack_tau_per_sample(vec, n_in: int, H: int):
    """Split a packed [..., (n_in + H + 2) H] row into (gW_in, gW_rec, gb, gtau)."""
    vec = np.asarray(vec)
    lead = vec.shape[:-1]
    a, c = H * n_in, H * n_in + H * H
    return (vec[..., :a].reshape(*lead, H, n_in), vec[..., a:c].reshape(*lead, H, H),
            vec[..., c:c + H], vec[..., c + H:c + 2 * H])
