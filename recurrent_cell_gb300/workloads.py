"""Named workloads and the seeded synthetic input generator.

This module holds no arithmetic of the CfC method: it only names the
workload shapes and draws random inputs.  Both the CUDA path (through the
Python binding) and the CPU oracle under ``oracle/`` are fed from here, so
the two sides always see the same fp32 (or bf16-valued) inputs.

Input recipe (fixed draw order, one ``numpy.random.default_rng(seed)``):

1. ``x``     [B, K, n_in]  ~ N(0, 1)
2. ``h0``    [B, n_hid]    ~ N(0, h0_std^2)   (std 1, or 0.5 for the large case)
3. ``W_in``  [3, n_hid, n_in]  ~ U(-1/sqrt(n_in), +1/sqrt(n_in))   heads f, g, h~
4. ``W_rec`` [3, n_hid, n_hid] ~ U(-1/sqrt(n_hid), +1/sqrt(n_hid))
5. ``y``     [B, n_hid]    ~ N(0, 1)          target of the loss 0.5*||h_K - y||^2
6. ``dt``    [B]           ~ U(0.5, 1.5) when ``dt_per_sample``; else the scalar 1.0
7. ``b``     [3, n_hid]    ~ U(-bias_scale, +bias_scale), drawn only when
   ``bias_scale > 0``; otherwise all zeros (the benchmark workloads)

Drawing ``b`` last keeps every other input of a seed the same whether or not
a bias is drawn.  The parity tests draw a nonzero bias (independent values
per head and unit) so that the kernels' bias loads and head offsets are
exercised; the benchmark workloads keep ``b = 0``.  When the workload stores activations and weights in
bf16, x, h0, W_in and W_rec are quantised to bf16 (round to nearest even)
after drawing; the arrays stay float32 but every value is bf16-exact.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

MATH_FP32 = 0
MATH_TF32 = 1
MATH_BF16 = 2
MATH_NAMES = {MATH_FP32: "fp32", MATH_TF32: "tf32", MATH_BF16: "bf16"}

GRAD_SCRATCH = 0
GRAD_GEMM = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    n_in: int
    n_hid: int
    math: int = MATH_FP32
    grad_path: int = GRAD_SCRATCH
    h0_std: float = 1.0
    dt_per_sample: bool = False
    seed: int = 0

    @property
    def N(self) -> int:
        """Packed per-sample parameter-gradient length 3*(n_in+n_hid+1)*n_hid."""
        return 3 * (self.n_in + self.n_hid + 1) * self.n_hid

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five configurations of the method's benchmark suite.
TINY = Workload("tiny_B4_K8_16x32_fp32", B=4, K=8, n_in=16, n_hid=32)
SMOKE = Workload("smoke_B32_K64_64x128_fp32", B=32, K=64, n_in=64, n_hid=128)
MID = Workload("mid_B1024_K64_64x128_tf32", B=1024, K=64, n_in=64, n_hid=128,
               math=MATH_TF32, grad_path=GRAD_GEMM)
LARGE = Workload("large_B8192_K8_128x256_bf16", B=8192, K=8, n_in=128, n_hid=256,
                 math=MATH_BF16, grad_path=GRAD_GEMM, h0_std=0.5, dt_per_sample=True)
WORKLOADS = {w.name: w for w in (TINY, SMOKE, MID, LARGE)}
SHORT_NAMES = {"tiny": TINY, "smoke": SMOKE, "mid": MID, "large": LARGE}

# Standalone reduce_axis0 cases: [B, N] fp32 ~ N(0, 1).
REDUCE_BATCHES = (32, 256, 1024)
REDUCE_TAILS = (40960, 40961)


def bf16_quantise(a: np.ndarray) -> np.ndarray:
    """Quantise float32 values to the nearest bf16 (ties to even), kept as float32.

    Used only to synthesise bf16-valued inputs.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def make_inputs(w: Workload, seed: int | None = None, bias_scale: float = 0.0) -> dict:
    """Draw the inputs of workload ``w`` (all float32 numpy arrays); ``b`` is
    U(+-bias_scale) per head and unit when ``bias_scale > 0``, else zero."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
    x = rng.standard_normal((B, K, n_in), dtype=np.float64).astype(np.float32)
    h0 = (rng.standard_normal((B, H), dtype=np.float64) * w.h0_std).astype(np.float32)
    a_in = 1.0 / np.sqrt(n_in)
    a_rec = 1.0 / np.sqrt(H)
    W_in = rng.uniform(-a_in, a_in, size=(3, H, n_in)).astype(np.float32)
    W_rec = rng.uniform(-a_rec, a_rec, size=(3, H, H)).astype(np.float32)
    y = rng.standard_normal((B, H), dtype=np.float64).astype(np.float32)
    if w.dt_per_sample:
        dt = rng.uniform(0.5, 1.5, size=(B,)).astype(np.float32)
    else:
        dt = np.full((1,), 1.0, dtype=np.float32)
    if bias_scale > 0:
        b = rng.uniform(-bias_scale, bias_scale, size=(3, H)).astype(np.float32)
    else:
        b = np.zeros((3, H), dtype=np.float32)
    if w.math == MATH_BF16:
        x, h0, W_in, W_rec = (bf16_quantise(a) for a in (x, h0, W_in, W_rec))
    return dict(x=x, h0=h0, W_in=W_in, W_rec=W_rec, b=b, dt=dt, y=y)


def make_reduce_input(B: int, N: int, seed: int = 0) -> np.ndarray:
    """[B, N] float32 ~ N(0, 1) for the standalone reduce_axis0 cases."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, N), dtype=np.float32)


# The pages' single-head tau-cell, FP32, on the tiny and smoke shapes: x, h0 ~
# N(0, 1); W_in ~ U(+-1/sqrt(n_in)), W_rec ~ U(+-1/sqrt(n_hid)); b = 0 (or
# U(+-bias_scale), drawn last); tau ~ U(0.5, 2.0) per unit; dt = 1.0 (or
# U(0.5, 1.5) per sample); y ~ N(0, 1).
TAU_TINY = Workload("tau_tiny_B4_K8_16x32_fp32", B=4, K=8, n_in=16, n_hid=32)
TAU_SMOKE = Workload("tau_smoke_B32_K64_64x128_fp32", B=32, K=64, n_in=64, n_hid=128)


def make_tau_inputs(w: Workload, seed: int | None = None, bias_scale: float = 0.0) -> dict:
    """Draw the inputs of a tau-cell workload (all float32 numpy arrays)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, K, n_in, H = w.B, w.K, w.n_in, w.n_hid
    x = rng.standard_normal((B, K, n_in), dtype=np.float64).astype(np.float32)
    h0 = (rng.standard_normal((B, H), dtype=np.float64) * w.h0_std).astype(np.float32)
    a_in, a_rec = 1.0 / np.sqrt(n_in), 1.0 / np.sqrt(H)
    W_in = rng.uniform(-a_in, a_in, size=(H, n_in)).astype(np.float32)
    W_rec = rng.uniform(-a_rec, a_rec, size=(H, H)).astype(np.float32)
    tau = rng.uniform(0.5, 2.0, size=(H,)).astype(np.float32)
    y = rng.standard_normal((B, H), dtype=np.float64).astype(np.float32)
    if w.dt_per_sample:
        dt = rng.uniform(0.5, 1.5, size=(B,)).astype(np.float32)
    else:
        dt = np.full((1,), 1.0, dtype=np.float32)
    if bias_scale > 0:
        b = rng.uniform(-bias_scale, bias_scale, size=(H,)).astype(np.float32)
    else:
        b = np.zeros((H,), dtype=np.float32)
    return dict(x=x, h0=h0, W_in=W_in, W_rec=W_rec, b=b, tau=tau, dt=dt, y=y)


# Multi-horizon GRN heads on the trunk rows, FP32.  The pages' shapes:
# HIDDEN = 128 (the CfC state), HEAD_MID = 64, 5 horizons, B = 32, K = 64
# (B*K = 2048 rows).  h ~ U(-1, 1) (a tanh-bounded state); weights
# Xavier-uniform with scale sqrt(1 / fan_in) as the pages initialise them
# (W1, w_skip: fan_in HIDDEN; W2, w_gate, w_main: fan_in HEAD_MID); biases
# ~ U(+-0.1) (the pages do not state theirs); grad_probs ~ N(0, 1) (dL/dp of a sum loss);
# lambda ~ U(0.5, 1.5) per horizon; grad_h_carry ~ N(0, 0.1).
@dataclass(frozen=True)
class GrnWorkload:
    name: str
    B: int
    K: int
    hidden: int = 128
    head_mid: int = 64
    n_horizons: int = 5
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.B * self.K


GRN_TINY = GrnWorkload("grn_tiny_B4_K8_32x16x3", B=4, K=8, hidden=32, head_mid=16, n_horizons=3)
GRN_SMOKE = GrnWorkload("grn_smoke_B32_K64_128x64x5", B=32, K=64)


def make_grn_inputs(w: GrnWorkload, seed: int | None = None) -> dict:
    """Draw the inputs of a GRN-heads workload (float32 numpy arrays); the
    parameter vector is packed in the documented order [W1 | b1 | W2 | b2 |
    w_gate | b_gate | w_main | b_main | w_skip | b_skip]."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    Hd, M, J, R = w.hidden, w.head_mid, w.n_horizons, w.rows
    sh, sm = np.sqrt(1.0 / Hd), np.sqrt(1.0 / M)
    sizes_scales = [(J * M * Hd, sh), (J * M, 0.1), (J * M * M, sm), (J * M, 0.1), (J * M, sm), (J, 0.1),
                    (J * M, sm), (J, 0.1), (J * Hd, sh), (J, 0.1)]
    params = np.concatenate([rng.uniform(-a, a, size=n) for n, a in sizes_scales]).astype(np.float32)
    h = rng.uniform(-1.0, 1.0, size=(R, Hd)).astype(np.float32)
    grad_probs = rng.standard_normal((R, J)).astype(np.float32)
    lam = rng.uniform(0.5, 1.5, size=(J,)).astype(np.float32)
    carry = (0.1 * rng.standard_normal((R, Hd))).astype(np.float32)
    return dict(h=h, params=params, grad_probs=grad_probs, lam=lam, carry=carry)
