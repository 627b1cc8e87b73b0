"""Pins of the oracle's reduce_axis0 (canonical float32 association order)."""

import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_reduce_golden():
    cases = []
    with open(os.path.join(GOLDEN, "reduce_axis0_order.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, B, rows, expect = [f.strip() for f in line.split(";")]
            B = int(B)
            col = np.zeros(B, dtype=np.float32)
            for item in rows.split():
                r, v = item.split("=")
                col[int(r)] = np.float32(float(v))
            cases.append((name, col, np.float32(float(expect))))
    return cases


@pytest.mark.parametrize("name, col, expect", load_reduce_golden())
def test_golden_order(name, col, expect):
    out = oracle.reduce_axis0(col.reshape(-1, 1))
    assert out.dtype == np.float32 and out.shape == (1,)
    assert out.view(np.uint32)[0] == np.array([expect], np.float32).view(np.uint32)[0], name


@pytest.mark.parametrize("B, N", [(1, 7), (5, 3), (256, 9), (257, 4), (300, 5), (1024, 6), (1031, 3)])
def test_integer_valued_sums_are_exact(B, N):
    """Small integers are exact in float32 and so are all their partial sums:
    the result must equal the exact integer column sum in any order."""
    b = np.arange(B)[:, None]
    j = np.arange(N)[None, :]
    a = (((7 * b + j) % 13) - 6).astype(np.float32)
    out = oracle.reduce_axis0(a)
    np.testing.assert_array_equal(out, a.astype(np.int64).sum(0).astype(np.float32))


def test_empty_batch_gives_zero():
    out = oracle.reduce_axis0(np.zeros((0, 5), np.float32))
    assert np.all(out.view(np.uint32) == 0)


@pytest.mark.parametrize("B", [1, 2, 255, 256, 300])
def test_negative_zero_columns_sum_to_positive_zero(B):
    """Every leaf starts from +0.0f, and +0.0f + (-0.0f) = +0.0f under round to
    nearest, so a column of -0.0 sums to +0.0 whatever B is; a sum that
    started from the first row instead would keep -0.0 once all 256 leaves
    hold one."""
    out = oracle.reduce_axis0(np.full((B, 3), -0.0, np.float32))
    assert np.all(out.view(np.uint32) == 0), B


def test_single_row_is_a_copy():
    a = np.random.default_rng(0).standard_normal((1, 100)).astype(np.float32)
    np.testing.assert_array_equal(oracle.reduce_axis0(a), a[0])


def _bitrev8(t):
    return int("{:08b}".format(t)[::-1], 2)


def test_equals_contiguous_tree_over_bit_reversed_leaves():
    """Equivalent form used by the CUDA reducer: leaf t holds the ordered
    stride-256 sum of rows t, t+256, ...; the stride-halving tree over t is the
    contiguous pairwise tree over leaves ordered by the 8-bit reversal of t."""
    rng = np.random.default_rng(9)
    for B in (3, 32, 100, 256, 700, 1024):
        a = rng.standard_normal((B, 17)).astype(np.float32)
        leaves = []
        for i in range(256):
            t = _bitrev8(i)
            acc = np.zeros(17, np.float32)
            for r in range(t, B, 256):
                acc = acc + a[r]
            leaves.append(acc)
        while len(leaves) > 1:
            leaves = [leaves[2 * m] + leaves[2 * m + 1] for m in range(len(leaves) // 2)]
        np.testing.assert_array_equal(oracle.reduce_axis0(a), leaves[0])


def test_close_to_float64_sum():
    a = np.random.default_rng(1).standard_normal((1024, 300)).astype(np.float32)
    np.testing.assert_allclose(oracle.reduce_axis0(a), a.astype(np.float64).sum(0), rtol=0, atol=2e-4)
