"""A float32 rendition of the CfC K loop with the CUDA kernels' rounding
points: the measuring instrument behind the reduced-precision tolerances of
the GPU parity tests.

TEST INSTRUMENT, not an oracle.  It computes what a correct float32
implementation with exactly the kernels' rounding points computes (numpy
float32 matrix products, i.e. fp32 accumulation in some order of the BLAS'
choosing), so its distance from the float64 oracle is the noise floor that
any such implementation (the GPU's included) must be allowed.  It shares no
code with the oracle or the CUDA path; its rounding helpers are written here
from the bit layouts.

Rounding points (the kernels' own, per precision mode):

* TF32: every operand of a contraction -- x_k, h_k, W_in, W_rec in the
  per-step projection; dA, W_rec, W_in in the carry and grad_x products; dA,
  x_k, h_k in the weight gradient -- is rounded to TF32 (low 13 bits of the
  binary32 pattern cleared, nearest, ties away from zero).  State,
  activations and accumulators stay float32.
* BF16: x, h0 and the weights arrive bf16-valued; the new state is rounded
  to bf16 (nearest even) and that value is stored and carried; dA is rounded
  to bf16 before every contraction it enters.
* FP32: no rounding.
"""

from __future__ import annotations

import numpy as np

FP32, TF32, BF16 = 0, 1, 2


def tf32(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


def bf16(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32).view(np.float32)


def kloop(inp: dict, mode: int, per_sample: bool = False) -> dict:
    """Forward + backward (loss 0.5*||h_K - y||^2) in float32; with
    per_sample, also the packed per-sample gradient rows
    [gW_in (c, i, j) | gW_rec (c, i, j) | gb (c, i)] of each sample's K rows."""
    f32 = np.float32
    opnd = {TF32: tf32, BF16: bf16}.get(mode, lambda a: np.asarray(a, dtype=f32))
    state = bf16 if mode == BF16 else (lambda a: np.asarray(a, dtype=f32))
    x = np.asarray(inp["x"], dtype=f32)
    B, K, n_in = x.shape
    H = inp["h0"].shape[1]
    Wi = opnd(np.asarray(inp["W_in"], dtype=f32).reshape(3 * H, n_in))
    Wr = opnd(np.asarray(inp["W_rec"], dtype=f32).reshape(3 * H, H))
    b = np.asarray(inp["b"], dtype=f32).reshape(1, 3 * H)
    dt = np.asarray(inp["dt"], dtype=f32).reshape(-1)
    dt = (np.full(B, dt[0], dtype=f32) if dt.size == 1 else dt)[:, None]
    y = np.asarray(inp["y"], dtype=f32)

    hs = np.empty((B, K + 1, H), dtype=f32)      # hs[:, k] = state entering step k
    hs[:, 0] = state(np.asarray(inp["h0"], dtype=f32))
    gate = np.empty((B, K, H), dtype=f32)
    g = np.empty_like(gate)
    hh = np.empty_like(gate)
    xo = opnd(x)
    for k in range(K):
        A = xo[:, k] @ Wi.T + opnd(hs[:, k]) @ Wr.T + b
        with np.errstate(over="ignore"):
            gate[:, k] = f32(1) / (f32(1) + np.exp(A[:, :H] * dt))
        g[:, k] = np.tanh(A[:, H:2 * H])
        hh[:, k] = np.tanh(A[:, 2 * H:])
        hs[:, k + 1] = state(gate[:, k] * g[:, k] + (f32(1) - gate[:, k]) * hh[:, k])

    carry = np.zeros((B, H), dtype=f32)
    dA = np.empty((B, K, 3 * H), dtype=f32)
    grad_x = np.empty((B, K, n_in), dtype=f32)
    for k in range(K - 1, -1, -1):
        delta = carry + (hs[:, K] - y if k == K - 1 else f32(0))
        gt, gg, hk = gate[:, k], g[:, k], hh[:, k]
        d = np.empty((B, 3 * H), dtype=f32)
        d[:, H:2 * H] = delta * gt * (f32(1) - gg * gg)
        d[:, 2 * H:] = delta * (f32(1) - gt) * (f32(1) - hk * hk)
        d[:, :H] = -dt * delta * (gg - hk) * gt * (f32(1) - gt)
        d = opnd(d)
        dA[:, k] = d
        grad_x[:, k] = d @ Wi
        carry = d @ Wr
    Zb = np.concatenate([xo, opnd(hs[:, :K]), np.ones((B, K, 1), dtype=f32)], axis=2)
    G = dA.reshape(B * K, 3 * H).T @ Zb.reshape(B * K, -1)
    out = dict(h_seq=hs[:, 1:], grad_W_in=G[:, :n_in].reshape(3, H, n_in),
               grad_W_rec=G[:, n_in:n_in + H].reshape(3, H, H), grad_b=G[:, n_in + H].reshape(3, H),
               grad_h0=carry, grad_x=grad_x)
    if per_sample:
        Gs = np.matmul(dA.transpose(0, 2, 1), Zb)                        # [B, 3H, n_in + H + 1]
        out["per_sample"] = np.concatenate([Gs[:, :, :n_in].reshape(B, -1), Gs[:, :, n_in:n_in + H].reshape(B, -1),
                                            Gs[:, :, n_in + H].reshape(B, -1)], axis=1)
    return out


def deviation(got: dict, ref: dict, rel: float, state_bf16: bool) -> dict:
    """Per output: normwise relative distance, and the smallest elementwise
    guard g (as a fraction of max|ref|) with |got - ref| <= rel|ref| + g max|ref|
    (plus one bf16 ulp, 2^-7|ref|, for a bf16-stored state)."""
    out = {}
    for k, r in ref.items():
        a = np.asarray(got[k], dtype=np.float64)
        r = np.asarray(r, dtype=np.float64)
        d = np.abs(a - r)
        allow = rel * np.abs(r) + (2.0 ** -7 * np.abs(r) if (state_bf16 and k == "h_seq") else 0.0)
        out[k] = dict(norm=float(np.linalg.norm(a - r) / np.linalg.norm(r)),
                      guard=float(max(0.0, (d - allow).max()) / np.abs(r).max()))
    return out
