"""CPU oracle for the batched CfC K-loop (forward, backward-through-time) and
for the deterministic column reducer ``reduce_axis0``.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the CPU
baseline leg of the benchmark may import or run this module.  It shares no
code with the CUDA path and never takes an input or an expected value from it.

Everything is plain numpy.  The cell arithmetic is float64; the reducer is
float32 in the exact association order of the pages' first reducer.

Sources (page title, section):

* "K-loop Parallelization Implementation Plan", Task 1 (reduce_axis0 kernel):
  [B, N] -> [N] column sums, overwrite; 256 threads stride over B starting
  from 0.0f, then a shared-memory tree with strides 128, 64, ..., 1.
* same page, Task 2 (cfc_step_batched forward): per-sample pre-activation
  b + W_in x_b + W_rec h_b with row-major [n_hid, n_in] / [n_hid, n_hid]
  weights and tanh as the squashing nonlinearity.
* same page, Task 3 (cfc_step_backward_batched): argument order, per-sample
  parameter-gradient scratch [B, ...] accumulated over the K loop and later
  summed over B, grad_x optional, grad_h_old overwrite.
* the three-head closed-form cell itself: heads f, g, h~ over
  W_in x + W_rec h + b; gate = sigmoid(-f * dt); h' = gate*g + (1-gate)*h~,
  with g = tanh, h~ = tanh and f the identity.
* "kernel-optimization" plan (2026-04-19), Task 2 Step 3: a weight gradient
  is the batch-dimension contraction  dW = Z^T dA  over all B*K rows.

Precision modes (the rounding points the CUDA path applies, mirrored here):

* FP32: no rounding.
* TF32: every operand of the projections and of the gradient contractions
  (x, h, W_in, W_rec and dA) is rounded to TF32 (10 explicit mantissa bits,
  round to nearest, ties away from zero); state and activations are not.
* BF16: x, h0, W_in, W_rec arrive bf16-valued; the new state h_{k+1} is
  rounded to bf16 (round to nearest even, through float32) and that rounded
  value is both stored and fed to the next step; dA is rounded to bf16
  before the gradient contractions.  Activations stay unrounded.
"""

from __future__ import annotations

import numpy as np

FP32, TF32, BF16 = 0, 1, 2


# --------------------------------------------------------------------------
# Rounding functions (from their definitions: IEEE binary32 bit layout).
# --------------------------------------------------------------------------

def round_bf16(a) -> np.ndarray:
    """Round to bfloat16 (8-bit significand), ties to even; input first taken
    to float32.  Returned as float64 holding the bf16 value."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def round_tf32(a) -> np.ndarray:
    """Round to TF32 (10 explicit significand bits: the low 13 bits of the
    binary32 pattern cleared), to nearest with ties away from zero; input
    first taken to float32.  Returned as float64."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x1000) & 0xFFFFE000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _operand(a, mode: int) -> np.ndarray:
    """A value as it enters a projection / gradient contraction."""
    if mode == TF32:
        return round_tf32(a)
    if mode == BF16:
        return round_bf16(a)
    return np.asarray(a, dtype=np.float64)


def _stored_state(h, mode: int) -> np.ndarray:
    """The new state as stored in h_seq and carried to the next step."""
    if mode == BF16:
        return round_bf16(h)
    return np.asarray(h, dtype=np.float64)


def _dt_vector(dt, B: int) -> np.ndarray:
    dt = np.asarray(dt, dtype=np.float64).reshape(-1)
    if dt.size == 1:
        return np.full(B, dt[0])
    assert dt.size == B, "dt must hold 1 or B values"
    return dt


# --------------------------------------------------------------------------
# Forward
# --------------------------------------------------------------------------

def cell_forward(x_k, h_k, W_in, W_rec, b, dt, mode: int = FP32):
    """One step of the three-head CfC cell for a batch of independent rows.

    x_k [n, n_in], h_k [n, H], W_in [3, H, n_in], W_rec [3, H, H], b [3, H],
    dt [n].  Returns (h_next [n, H], gate, g, hh) with
      A_c   = b_c + W_in[c] x_k + W_rec[c] h_k           (c = f, g, h~)
      g     = tanh(A_g),  hh = tanh(A_h~),  gate = 1 / (1 + exp(A_f * dt))
      h_next = gate * g + (1 - gate) * hh
    """
    xo = _operand(x_k, mode)
    ho = _operand(h_k, mode)
    Wi = _operand(W_in, mode)
    Wr = _operand(W_rec, mode)
    n = xo.shape[0]
    H = Wr.shape[1]
    # A[n, c, i] = b[c, i] + sum_j W_in[c, i, j] x[n, j] + sum_j W_rec[c, i, j] h[n, j]
    A = (np.asarray(b, dtype=np.float64).reshape(1, 3 * H)
         + xo @ Wi.reshape(3 * H, -1).T + ho @ Wr.reshape(3 * H, H).T).reshape(n, 3, H)
    f = A[:, 0]
    g = np.tanh(A[:, 1])
    hh = np.tanh(A[:, 2])
    with np.errstate(over="ignore"):
        gate = 1.0 / (1.0 + np.exp(f * np.asarray(dt, dtype=np.float64)[:, None]))
    h_next = gate * g + (1.0 - gate) * hh
    return _stored_state(h_next, mode), gate, g, hh


def forward(x, h0, W_in, W_rec, b, dt, mode: int = FP32) -> dict:
    """K-loop forward.  h_seq[:, k] = h_{k+1} (h0 itself is not repeated)."""
    x = np.asarray(x)
    B, K, _ = x.shape
    H = np.asarray(h0).shape[1]
    dtv = _dt_vector(dt, B)
    h = _stored_state(np.asarray(h0, dtype=np.float64), mode)
    h_seq = np.empty((B, K, H))
    gates = np.empty((B, K, H))
    gs = np.empty((B, K, H))
    hhs = np.empty((B, K, H))
    for k in range(K):
        h, gate, g, hh = cell_forward(x[:, k], h, W_in, W_rec, b, dtv, mode)
        h_seq[:, k] = h
        gates[:, k], gs[:, k], hhs[:, k] = gate, g, hh
    return dict(h_seq=h_seq, gate=gates, g=gs, hh=hhs)


# --------------------------------------------------------------------------
# Backward through time
# --------------------------------------------------------------------------

def per_sample_length(n_in: int, H: int) -> int:
    """Packed per-sample gradient length N = 3*(n_in + H + 1)*H."""
    return 3 * (n_in + H + 1) * H


def backward(x, h0, W_in, W_rec, b, dt, mode: int = FP32,
             grad_h_seq=None, grad_h_last=None, y=None, per_sample: bool = True) -> dict:
    """Backward through the K loop.

    Upstream gradient of h_seq[:, k] is grad_h_seq[:, k] (optional); the last
    state additionally receives grad_h_last (optional) and, when a target y
    is given, the gradient of 0.5*||h_K - y||^2, i.e. h_K - y.

    Per step k = K-1 .. 0 with delta = carry + upstream:
      dA_g = delta * gate * (1 - g^2)
      dA_h = delta * (1 - gate) * (1 - hh^2)
      dA_f = -dt * delta * (g - hh) * gate * (1 - gate)
      carry      = sum_c W_rec[c]^T dA_c
      grad_x[k]  = sum_c W_in[c]^T  dA_c
    grad_h0 = carry after step 0.  The parameter gradients are the sums over
    all rows r = (b, k) of the outer products dA_r (x) [x_r; h_r; 1]:
      gW_in[c] = sum dA_c (x) x_k,  gW_rec[c] = sum dA_c (x) h_k,  gb[c] = sum dA_c
    taken as one matrix product over the B*K rows (the batch-dimension GEMM of
    the "kernel-optimization" plan, Task 2 Step 3) and, per sample, over that
    sample's K rows.

    Returns ``grad_W_in`` [3, H, n_in], ``grad_W_rec`` [3, H, H], ``grad_b``
    [3, H] (float64 sums over the batch), ``grad_h0`` [B, H], ``grad_x``
    [B, K, n_in], ``h_seq``, ``dA`` [B, K, 3, H] and, if ``per_sample``, the
    packed per-sample gradients ``per_sample`` [B, N] laid out as
    [gW_in (c, i, j) | gW_rec (c, i, j) | gb (c, i)].
    """
    x = np.asarray(x)
    B, K, n_in = x.shape
    H = np.asarray(h0).shape[1]
    dtv = _dt_vector(dt, B)
    fw = forward(x, h0, W_in, W_rec, b, dt, mode)
    h_seq = fw["h_seq"]
    h_prev = np.concatenate(
        [_stored_state(np.asarray(h0, dtype=np.float64), mode)[:, None], h_seq[:, :-1]], axis=1)

    Wi = _operand(W_in, mode).reshape(3 * H, n_in)
    Wr = _operand(W_rec, mode).reshape(3 * H, H)
    grad_x = np.zeros((B, K, n_in))
    dA_all = np.zeros((B, K, 3, H))
    carry = np.zeros((B, H))
    for k in range(K - 1, -1, -1):
        delta = carry.copy()
        if grad_h_seq is not None:
            delta += np.asarray(grad_h_seq, dtype=np.float64)[:, k]
        if k == K - 1:
            if grad_h_last is not None:
                delta += np.asarray(grad_h_last, dtype=np.float64)
            if y is not None:
                delta += h_seq[:, K - 1] - np.asarray(y, dtype=np.float64)
        gate, g, hh = fw["gate"][:, k], fw["g"][:, k], fw["hh"][:, k]
        dA = np.empty((B, 3, H))
        dA[:, 1] = delta * gate * (1.0 - g * g)
        dA[:, 2] = delta * (1.0 - gate) * (1.0 - hh * hh)
        dA[:, 0] = -dtv[:, None] * delta * (g - hh) * gate * (1.0 - gate)
        dAo = _operand(dA, mode)
        dA_all[:, k] = dAo
        grad_x[:, k] = dAo.reshape(B, 3 * H) @ Wi
        carry = dAo.reshape(B, 3 * H) @ Wr

    # rows r = (b, k): z_r = [x_r; h_r; 1] as contraction operands
    Z = np.concatenate([_operand(x, mode), _operand(h_prev, mode), np.ones((B, K, 1))], axis=2)
    D = dA_all.reshape(B, K, 3 * H)
    G = D.reshape(B * K, 3 * H).T @ Z.reshape(B * K, n_in + H + 1)       # [3H, n_in + H + 1]
    out = dict(grad_W_in=G[:, :n_in].reshape(3, H, n_in),
               grad_W_rec=G[:, n_in:n_in + H].reshape(3, H, H),
               grad_b=G[:, n_in + H].reshape(3, H),
               grad_h0=carry, grad_x=grad_x, h_seq=h_seq, dA=dA_all)
    if per_sample:
        Gs = np.matmul(D.transpose(0, 2, 1), Z)                           # [B, 3H, n_in + H + 1]
        out["per_sample"] = np.concatenate(
            [Gs[:, :, :n_in].reshape(B, -1), Gs[:, :, n_in:n_in + H].reshape(B, -1),
             Gs[:, :, n_in + H].reshape(B, -1)], axis=1)
    return out


def unpack_per_sample(vec, n_in: int, H: int):
    """Split a packed [..., N] gradient into (gW_in, gW_rec, gb)."""
    vec = np.asarray(vec)
    n1, n2 = 3 * H * n_in, 3 * H * H
    lead = vec.shape[:-1]
    return (vec[..., :n1].reshape(*lead, 3, H, n_in),
            vec[..., n1:n1 + n2].reshape(*lead, 3, H, H),
            vec[..., n1 + n2:].reshape(*lead, 3, H))


# --------------------------------------------------------------------------
# reduce_axis0: the canonical float32 association order
# --------------------------------------------------------------------------

REDUCE_THREADS = 256


def reduce_axis0(per_batch) -> np.ndarray:
    """[B, N] float32 -> [N] float32, OVERWRITE semantics, in the association
    order of the pages' first reducer (one 256-thread block per column):

      p[t] = ((0.0f + in[t]) + in[t+256]) + in[t+512] + ...   (t = 0..255)
      for s = 128, 64, ..., 1:  p[t] = p[t] + p[t+s]   for t < s
      out  = p[0]

    All additions are float32 with round-to-nearest-even (numpy elementwise).
    """
    a = np.ascontiguousarray(per_batch, dtype=np.float32)
    assert a.ndim == 2
    B, N = a.shape
    T = REDUCE_THREADS
    p = np.zeros((T, N), dtype=np.float32)
    for t in range(min(B, T)):
        acc = np.zeros(N, dtype=np.float32)
        for bi in range(t, B, T):
            acc = acc + a[bi]          # float32 + float32 -> float32
        p[t] = acc
    s = T // 2
    while s > 0:
        p[:s] = p[:s] + p[s:2 * s]
        s //= 2
    return p[0].copy()
