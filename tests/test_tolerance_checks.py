"""The comparison every GPU parity test ends in (gpu_common.assert_close) is
not vacuous: it accepts differences inside the stated tolerances and rejects
differences just outside them, non-finite values and shape mismatches.
CPU only (the helper takes host arrays)."""

import numpy as np
import pytest

from gpu_common import FP32_ABS, FP32_REL, LP_REL, assert_close
from recurrent_cell_gb300 import workloads as wl


def _ref():
    return np.random.default_rng(0).standard_normal(1000)


def test_fp32_elementwise_bound():
    ref = _ref()
    tol = FP32_ABS + FP32_REL * np.abs(ref)
    assert_close(ref + 0.99 * tol, ref, wl.MATH_FP32, "inside")
    bad = ref.copy()
    bad[123] += 1.01 * tol[123]
    with pytest.raises(AssertionError, match="1 of 1000 elements"):
        assert_close(bad, ref, wl.MATH_FP32, "one element outside")


@pytest.mark.parametrize("math", [wl.MATH_TF32, wl.MATH_BF16])
def test_reduced_precision_normwise_bound(math):
    ref = _ref()
    d = np.random.default_rng(1).standard_normal(ref.size)
    d *= np.linalg.norm(ref) / np.linalg.norm(d)
    assert_close(ref + 0.9 * LP_REL * d, ref, math, "inside")
    with pytest.raises(AssertionError, match="normwise"):
        assert_close(ref + 1.1 * LP_REL * d, ref, math, "outside")


def test_reduced_precision_guard_catches_one_wrong_element():
    """A single element far off keeps the normwise error small on a large
    tensor, but the elementwise guard still rejects it."""
    ref = np.random.default_rng(2).standard_normal(200000)
    bad = ref.copy()
    bad[7] += 0.05 * np.abs(ref).max()
    assert np.linalg.norm(bad - ref) < LP_REL * np.linalg.norm(ref)
    with pytest.raises(AssertionError, match="out of tolerance"):
        assert_close(bad, ref, wl.MATH_BF16, "isolated")


def test_non_finite_and_shape_mismatch_fail():
    ref = _ref()
    bad = ref.copy()
    bad[0] = np.nan
    with pytest.raises(AssertionError, match="non-finite"):
        assert_close(bad, ref, wl.MATH_FP32, "nan")
    with pytest.raises(AssertionError):
        assert_close(ref[:-1], ref, wl.MATH_FP32, "shape")
