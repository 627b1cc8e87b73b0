"""Planted mistakes in copies of the CPU oracle: each must fail at least one pin.

Every mutant is one plausible slip in the oracle's source text (a dropped term,
a flipped sign, a wrong index or step, a transposed operand, a wrong
association order or rounding rule).  The mutated text is loaded as a module
of its own, the pin tests are pointed at it, and at least one of them has to
fail.  The oracle files themselves are never changed; the unmutated copy must
pass every pin (so the harness really runs them).  CPU only.
"""

import os
import types

import pytest

import test_grn_oracle_pins as grn_pins
import test_oracle_pins as cfc_pins
import test_reduce_oracle as reduce_pins
import test_tau_oracle_pins as tau_pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def load_copy(filename, old=None, new=None):
    """The oracle file `filename` as a fresh module, with `old` replaced by
    `new` (which must occur exactly once) when given."""
    path = os.path.join(ORACLE_DIR, filename)
    with open(path) as fh:
        src = fh.read()
    if old is not None:
        assert src.count(old) == 1, f"{filename}: the mutated text must occur exactly once: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("mutant_" + filename[:-3])
    mod.__file__ = path
    exec(compile(src, f"{path} (copy)", "exec"), mod.__dict__)
    return mod


# ------------------------------------------------------------------ the pins

def cfc_checks(m):
    """(name, callable) pairs running the cell and reducer pins against m;
    the slow ones last."""
    p, r = cfc_pins, reduce_pins
    checks = [
        ("scalar step golden", p.test_scalar_step_golden),
        ("zero weights K=1", lambda: p.test_zero_weights_closed_form(1)),
        ("zero weights K=3", lambda: p.test_zero_weights_closed_form(3)),
        ("dt = 0", p.test_dt_zero_freezes_gate),
        ("batch independence", p.test_batch_rows_independent_and_permutation_equivariant),
        ("reduced = sum of rows", p.test_reduced_gradient_is_sum_of_per_sample),
        ("tf32 definition", p.test_tf32_rounding_definition),
        ("bf16 rounding points", lambda: p.test_mode_rounding_points_single_step(m.BF16, m.round_bf16)),
        ("tf32 rounding points", lambda: p.test_mode_rounding_points_single_step(m.TF32, m.round_tf32)),
        ("bf16 operands", lambda: p.test_mode_rounds_every_contraction_operand(m.BF16, m.round_bf16)),
        ("tf32 operands", lambda: p.test_mode_rounds_every_contraction_operand(m.TF32, m.round_tf32)),
        ("reduce: integer sums", lambda: r.test_integer_valued_sums_are_exact(1031, 3)),
        ("reduce: empty", r.test_empty_batch_gives_zero),
        ("reduce: copy", r.test_single_row_is_a_copy),
        ("reduce: -0.0 columns", lambda: [r.test_negative_zero_columns_sum_to_positive_zero(b) for b in (2, 256)]),
        ("reduce: bit-reversed tree", r.test_equals_contiguous_tree_over_bit_reversed_leaves),
    ]
    for name, col, expect in r.load_reduce_golden():
        checks.append((f"reduce golden {name}", lambda n=name, c=col, e=expect: r.test_golden_order(n, c, e)))
    checks += [
        ("Elman RNN, gate 0", lambda: p.test_saturated_gate_is_elman_rnn(10.0, 2)),
        ("Elman RNN, gate 1", lambda: p.test_saturated_gate_is_elman_rnn(-10.0, 1)),
        ("bf16 vs torch", p.test_bf16_rounding_matches_torch_conversion),
        ("finite differences", p.test_finite_differences_every_element_tiny),
    ]
    return checks


def tau_checks(m):
    p = tau_pins
    checks = [
        ("zero weights", p.test_zero_weights_closed_form),
        ("tau below clamp", p.test_tau_below_clamp_is_the_tanh_rnn),
        ("huge tau", p.test_huge_tau_keeps_the_state),
        ("independence", p.test_samples_are_independent_and_rows_sum_to_the_batch_gradient),
        ("clamped tau, live decay", p.test_clamped_tau_gets_no_gradient_while_its_decay_is_live),
        ("clamp value", p.test_clamp_value_in_the_closed_form),
    ]
    for name in ("W_in", "W_rec", "b", "tau", "h0", "x"):
        checks.append((f"finite differences {name}", lambda n=name: p.test_gradients_match_central_differences(n)))
    return checks


def grn_checks(m):
    p = grn_pins
    return [
        ("parameter count", p.test_param_length_matches_the_pages_count),
        ("normal CDF", p.test_gelu_against_printed_normal_cdf),
        ("lambda zero", p.test_lambda_zero_returns_the_carry_and_leaves_parameter_gradients),
        ("zero first layer", p.test_zero_first_layer_closed_form),
        ("independence", p.test_samples_are_independent_and_rows_sum_to_the_batch_gradient),
        ("segment order", p.test_pack_unpack_round_trip_and_segment_order),
        ("finite differences, parameters", p.test_parameter_gradient_matches_central_differences),
        ("finite differences, trunk h0", lambda: p.test_trunk_gradient_per_horizon_is_lambda_scaled(0)),
        ("finite differences, trunk h1", lambda: p.test_trunk_gradient_per_horizon_is_lambda_scaled(1)),
    ]


# (module file, pin module, attribute the pins read the oracle from, checks)
TARGETS = {
    "cfc_oracle.py": ([cfc_pins, reduce_pins], "oracle", cfc_checks),
    "tau_oracle.py": ([tau_pins], "to", tau_checks),
    "grn_oracle.py": ([grn_pins], "go", grn_checks),
}


def first_failure(monkeypatch, filename, mod):
    """Name of the first pin that fails against `mod`, or None."""
    pin_modules, attr, checks = TARGETS[filename]
    for pm in pin_modules:
        monkeypatch.setattr(pm, attr, mod)
    for name, check in checks(mod):
        try:
            check()
        except (Exception, pytest.fail.Exception):
            return name
    return None


# ------------------------------------------------------------------ mutants

MUTANTS = [
    # three-head cell, forward
    ("cfc_oracle.py", "gate sign", "np.exp(f * np.asarray(dt", "np.exp(-f * np.asarray(dt"),
    ("cfc_oracle.py", "heads swapped in the mix",
     "h_next = gate * g + (1.0 - gate) * hh", "h_next = gate * hh + (1.0 - gate) * g"),
    ("cfc_oracle.py", "g head without tanh", "g = np.tanh(A[:, 1])", "g = A[:, 1]"),
    ("cfc_oracle.py", "W_rec transposed in the projection",
     "ho @ Wr.reshape(3 * H, H).T", "ho @ Wr.transpose(0, 2, 1).reshape(3 * H, H).T"),
    ("cfc_oracle.py", "bias dropped",
     "A = (np.asarray(b, dtype=np.float64)", "A = (0.0 * np.asarray(b, dtype=np.float64)"),
    ("cfc_oracle.py", "heads interleaved per unit instead of head-major",
     ".T).reshape(n, 3, H)", ".T).reshape(n, H, 3).transpose(0, 2, 1)"),
    ("cfc_oracle.py", "h~ head reads the g pre-activation", "hh = np.tanh(A[:, 2])", "hh = np.tanh(A[:, 1])"),
    # backward
    ("cfc_oracle.py", "grad_x written at the mirrored step",
     "grad_x[:, k] = dAo.reshape(B, 3 * H) @ Wi", "grad_x[:, K - 1 - k] = dAo.reshape(B, 3 * H) @ Wi"),
    ("cfc_oracle.py", "dA_g without tanh'",
     "dA[:, 1] = delta * gate * (1.0 - g * g)", "dA[:, 1] = delta * gate"),
    ("cfc_oracle.py", "dA_h with gate for 1 - gate",
     "dA[:, 2] = delta * (1.0 - gate) * (1.0 - hh * hh)", "dA[:, 2] = delta * gate * (1.0 - hh * hh)"),
    ("cfc_oracle.py", "dA_f sign", "dA[:, 0] = -dtv[:, None] * delta", "dA[:, 0] = dtv[:, None] * delta"),
    ("cfc_oracle.py", "dA_f without dt",
     "dA[:, 0] = -dtv[:, None] * delta * (g - hh)", "dA[:, 0] = -delta * (g - hh)"),
    ("cfc_oracle.py", "carry through W_rec untransposed",
     "carry = dAo.reshape(B, 3 * H) @ Wr",
     "carry = dAo.reshape(B, 3 * H) @ Wr.reshape(3, H, H).transpose(0, 2, 1).reshape(3 * H, H)"),
    ("cfc_oracle.py", "carry dropped", "delta = carry.copy()", "delta = 0.0 * carry"),
    ("cfc_oracle.py", "per-step upstream gradient at the mirrored step",
     "np.asarray(grad_h_seq, dtype=np.float64)[:, k]",
     "np.asarray(grad_h_seq, dtype=np.float64)[:, K - 1 - k]"),
    ("cfc_oracle.py", "loss gradient sign",
     "delta += h_seq[:, K - 1] - np.asarray(y, dtype=np.float64)",
     "delta += np.asarray(y, dtype=np.float64) - h_seq[:, K - 1]"),
    ("cfc_oracle.py", "weight gradient against h_{k+1} instead of h_k",
     "_operand(h_prev, mode), np.ones", "_operand(h_seq, mode), np.ones"),
    ("cfc_oracle.py", "per-sample segments swapped",
     "[Gs[:, :, :n_in].reshape(B, -1), Gs[:, :, n_in:n_in + H].reshape(B, -1),",
     "[Gs[:, :, n_in:n_in + H].reshape(B, -1), Gs[:, :, :n_in].reshape(B, -1),"),
    # precision modes
    ("cfc_oracle.py", "bf16 state not rounded", "return round_bf16(h)", "return np.asarray(h, dtype=np.float64)"),
    ("cfc_oracle.py", "dA not rounded", "dAo = _operand(dA, mode)", "dAo = dA"),
    ("cfc_oracle.py", "W_in not rounded in the projection",
     "Wi = _operand(W_in, mode)\n", "Wi = np.asarray(W_in, dtype=np.float64)\n"),
    ("cfc_oracle.py", "state operand not rounded in the projection",
     "ho = _operand(h_k, mode)", "ho = np.asarray(h_k, dtype=np.float64)"),
    ("cfc_oracle.py", "W_in not rounded in grad_x",
     "Wi = _operand(W_in, mode).reshape(3 * H, n_in)", "Wi = np.asarray(W_in, dtype=np.float64).reshape(3 * H, n_in)"),
    ("cfc_oracle.py", "x not rounded in the weight gradient",
     "Z = np.concatenate([_operand(x, mode)", "Z = np.concatenate([np.asarray(x, dtype=np.float64)"),
    ("cfc_oracle.py", "bf16 ties away from zero", "lsb = (u >> 16) & 1", "lsb = 0 * u"),
    ("cfc_oracle.py", "tf32 truncation", "u = (u + 0x1000) & 0xFFFFE000", "u = u & 0xFFFFE000"),
    ("cfc_oracle.py", "first sample's dt for every sample", "    return dt\n", "    return np.full(B, dt[0])\n"),
    ("cfc_oracle.py", "last-step seeds added at every step", "        if k == K - 1:\n", "        if True:\n"),
    ("cfc_oracle.py", "weight gradient's h_k shifted by one step",
     "h_seq[:, :-1]], axis=1)", "h_seq[:, 1:]], axis=1)"),
    # reducer order
    ("cfc_oracle.py", "leaf rows in descending order",
     "for bi in range(t, B, T):", "for bi in reversed(range(t, B, T)):"),
    ("cfc_oracle.py", "tree pairs adjacent leaves",
     "p[:s] = p[:s] + p[s:2 * s]", "p[:s] = p[0:2 * s:2] + p[1:2 * s:2]"),
    ("cfc_oracle.py", "128 leaves", "T = REDUCE_THREADS", "T = REDUCE_THREADS // 2"),
    ("cfc_oracle.py", "leaf sums start from -0.0",
     "acc = np.zeros(N, dtype=np.float32)", "acc = np.full(N, -0.0, dtype=np.float32)"),
    # tau cell
    ("tau_oracle.py", "decay sign", "np.exp(-np.asarray(dt_b", "np.exp(np.asarray(dt_b"),
    ("tau_oracle.py", "decay and input weight swapped",
     "h = h * d + (1.0 - d) * s", "h = h * (1.0 - d) + d * s"),
    ("tau_oracle.py", "d_pre without 1 - decay",
     "d_pre = dh * (1.0 - d) * (1.0 - s * s)", "d_pre = dh * (1.0 - s * s)"),
    ("tau_oracle.py", "carry without the decay path", "carry = d_pre @ Wr + dh * d", "carry = d_pre @ Wr"),
    ("tau_oracle.py", "carry through W_rec^T", "carry = d_pre @ Wr + dh * d", "carry = d_pre @ Wr.T + dh * d"),
    ("tau_oracle.py", "grad_tau sign", "dh * (hp - s) * d", "dh * (s - hp) * d"),
    ("tau_oracle.py", "clamp ignored in grad_tau", "np.where(live[None, :], ", "np.where(True, "),
    ("tau_oracle.py", "clamp at 1e-3", "TAU_EPS = 1e-6", "TAU_EPS = 1e-3"),
    ("tau_oracle.py", "clamp at 1e-9", "TAU_EPS = 1e-6", "TAU_EPS = 1e-9"),
    ("tau_oracle.py", "gradient mask at tau >= eps", "live = tau > TAU_EPS", "live = tau >= TAU_EPS"),
    ("tau_oracle.py", "first sample's dt for every sample",
     "return np.full(B, dt[0]) if dt.size == 1 else dt", "return np.full(B, dt[0])"),
    ("tau_oracle.py", "last-step seeds added at every step", "        if k == K - 1:\n", "        if True:\n"),
    # GRN heads
    ("grn_oracle.py", "GELU with the wrong CDF scale",
     "return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))", "return 0.5 * z * (1.0 + erf(z))"),
    ("grn_oracle.py", "gate not squashed",
     "logit = skip + sigmoid(gate) * main\n    return", "logit = skip + gate * main\n    return"),
    ("grn_oracle.py", "dgate without sigmoid'",
     'dgate = dlogit * f["main"] * sg * (1.0 - sg)', 'dgate = dlogit * f["main"] * sg'),
    ("grn_oracle.py", "lambda applied to the carry",
     "grad_h = grad_h + np.asarray(grad_h_carry, dtype=np.float64)",
     "grad_h = grad_h + lam.sum() * np.asarray(grad_h_carry, dtype=np.float64)"),
    ("grn_oracle.py", "W2 transposed in the backward",
     'da1 = np.einsum("jmn,rjm->rjn", P["W2"], dz2)', 'da1 = np.einsum("jnm,rjm->rjn", P["W2"], dz2)'),
    ("grn_oracle.py", "skip path dropped from the trunk gradient",
     ' + dskip[:, :, None] * P["w_skip"][None]', ""),
    ("grn_oracle.py", "b1 dropped", 'P["W1"], h) + P["b1"][None]', 'P["W1"], h)'),
    ("grn_oracle.py", "sigmoid' dropped from dlogit", "dlogit = gp * p * (1.0 - p)", "dlogit = gp * p"),
    ("grn_oracle.py", "gate and main weights swapped in dz2",
     'dmain[:, :, None] * P["w_main"][None] + dgate[:, :, None] * P["w_gate"][None]',
     'dmain[:, :, None] * P["w_gate"][None] + dgate[:, :, None] * P["w_main"][None]'),
    ("grn_oracle.py", "skip term halved", 'skip = h @ P["w_skip"].T', 'skip = h @ P["w_skip"].T * 0.5'),
    ("grn_oracle.py", "rows taken step-major",
     "per_row = pack_grn(rows, Hd, M, J).reshape(B, K, -1)",
     "per_row = pack_grn(rows, Hd, M, J).reshape(K, B, -1).transpose(1, 0, 2)"),
]


@pytest.mark.parametrize("filename", sorted(TARGETS))
def test_unmutated_copy_passes_every_pin(monkeypatch, filename):
    assert first_failure(monkeypatch, filename, load_copy(filename)) is None


@pytest.mark.parametrize("filename, what, old, new", MUTANTS, ids=[m[1] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, filename, what, old, new):
    caught = first_failure(monkeypatch, filename, load_copy(filename, old, new))
    assert caught is not None, f"no pin catches the planted mistake '{what}' in {filename}"
