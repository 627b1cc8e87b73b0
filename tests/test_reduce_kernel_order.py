"""The association order of the CUDA reducer's design, modelled on the CPU in
float32 and compared bit for bit with the oracle's canonical order (CPU only).

The kernel (reduce_axis0.cu) does not sum in the canonical loop order: warp w
of a block owns a 32-leaf subtree, its lanes are split into LG groups of LPG
leaves each, leaves are visited by their 8-bit bit-reversed index, small
batches visit only NL = 8 * LG * LPG leaves, and the partial sums meet by
shuffles and in shared memory.  This model follows those steps literally for
every kernel configuration (VEC only changes how many columns a lane holds,
not the order), so the design argument -- that this is the canonical tree --
is checked here for every batch band; the GPU tests check the kernel itself.
"""

import numpy as np
import pytest

import oracle

# (LG, LPG) per configuration, as the launcher picks them for a batch size:
# float4 rows and scalar rows have their own tables.
VEC_CFG = {0: (4, 8), 1: (4, 4), 2: (4, 2), 3: (4, 1)}
SCALAR_CFG = {0: (4, 8), 1: (1, 16), 2: (1, 8), 3: (1, 4)}
WARPS = 8


def band(B):
    return 0 if B > 128 else 1 if B > 64 else 2 if B > 32 else 3


def rev8(i):
    return int(f"{i:08b}"[::-1], 2)


def model(a, LG, LPG):
    """Column sums of a [B, N] float32 matrix in the kernel's order."""
    a = np.asarray(a, np.float32)
    B, N = a.shape
    NL = WARPS * LG * LPG
    LS = 256 // NL
    zero = np.zeros(N, np.float32)
    part = []
    for w in range(WARPS):
        group_totals = []
        for lg in range(LG):
            v = []
            for m in range(LPG):
                t = rev8(((w * LG + lg) * LPG + m) * LS)
                acc = (zero + a[t]) if t < B else zero.copy()
                if NL == 256:
                    off = 256
                    while off < B:
                        if t + off < B:
                            acc = acc + a[t + off]
                        off += 256
                v.append(acc)
            width = 1
            while width < LPG:                         # the lane group's pairwise subtree
                for m in range(0, LPG - width, 2 * width):
                    v[m] = v[m] + v[m + width]
                width *= 2
            group_totals.append(v[0])
        g = group_totals                               # ((g0 + g1) + (g2 + g3)) by shuffles
        if LG == 4:
            total = (g[0] + g[1]) + (g[2] + g[3])
        elif LG == 2:
            total = g[0] + g[1]
        else:
            total = g[0]
        part.append(total)
    p = part                                           # the 8 warps' subtrees in shared memory
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]))


@pytest.mark.parametrize("table", ["vec", "scalar"])
@pytest.mark.parametrize("B", [1, 2, 5, 31, 32, 33, 47, 64, 65, 100, 128, 129, 200, 256, 257, 511, 700, 1024, 1031])
def test_kernel_order_is_the_canonical_order(B, table):
    LG, LPG = (VEC_CFG if table == "vec" else SCALAR_CFG)[band(B)]
    rng = np.random.default_rng(B)
    # magnitudes spread over many binades so that any change of association shows in the bits
    a = (rng.standard_normal((B, 24)) * np.exp2(rng.integers(-12, 12, (B, 24)))).astype(np.float32)
    want = oracle.reduce_axis0(a)
    got = model(a, LG, LPG)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_model_detects_a_wrong_order():
    """The comparison above can fail: pairing the lane groups in another order
    (g0 + g2) + (g1 + g3) changes the bits on the same kind of data."""
    rng = np.random.default_rng(0)
    a = (rng.standard_normal((1024, 64)) * np.exp2(rng.integers(-12, 12, (1024, 64)))).astype(np.float32)
    want = oracle.reduce_axis0(a).view(np.uint32)
    LG, LPG = VEC_CFG[0]
    NL = WARPS * LG * LPG
    perm = [rev8(i) for i in range(256)]
    leaves = []
    for i in range(256):
        t = perm[i]
        acc = np.zeros(64, np.float32)
        for r in range(t, 1024, 256):
            acc = acc + a[r]
        leaves.append(acc)
    # regroup the 32-leaf subtree of each warp as (g0 + g2) + (g1 + g3)
    def subtree(xs):
        while len(xs) > 1:
            xs = [xs[2 * k] + xs[2 * k + 1] for k in range(len(xs) // 2)]
        return xs[0]
    parts = []
    for w in range(WARPS):
        g = [subtree(leaves[w * 32 + 8 * q: w * 32 + 8 * q + 8]) for q in range(4)]
        parts.append((g[0] + g[2]) + (g[1] + g[3]))
    wrong = ((parts[0] + parts[1]) + (parts[2] + parts[3])) + ((parts[4] + parts[5]) + (parts[6] + parts[7]))
    assert NL == 256 and np.any(wrong.view(np.uint32) != want)
