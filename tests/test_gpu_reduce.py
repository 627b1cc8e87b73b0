"""reduce_axis0 on the GPU, through the C ABI, against the oracle: bit-exact."""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import workloads as wl
from gpu_common import require_gpu, dev, torch_mod
from test_reduce_oracle import load_reduce_golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def gpu_reduce(a, out_offset=0, in_offset=0):
    """Run reduce_axis0 with optional element offsets of the input/output
    inside larger buffers; the guard regions around the output are checked
    to be untouched."""
    torch = torch_mod()
    B, N = a.shape
    flat = np.full(in_offset + B * N, np.nan, np.float32)
    flat[in_offset:] = a.reshape(-1)
    src = dev(flat)
    per_batch = src[in_offset:].view(B, N)
    guard = 64
    out_buf = torch.full((out_offset + N + guard,), float("nan"), device="cuda")
    out = out_buf[out_offset:out_offset + N]
    cfc.reduce_axis0(per_batch, out)
    host = out_buf.cpu().numpy()
    assert np.all(np.isnan(host[:out_offset])) and np.all(np.isnan(host[out_offset + N:])), \
        "reduce_axis0 wrote outside its output"
    return host[out_offset:out_offset + N].copy()


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("B", wl.REDUCE_BATCHES)
@pytest.mark.parametrize("N", wl.REDUCE_TAILS)
def test_standalone_configs_bit_exact(B, N):
    a = wl.make_reduce_input(B, N, seed=B + N)
    got = gpu_reduce(a)
    np.testing.assert_array_equal(bits(got), bits(oracle.reduce_axis0(a)))


@pytest.mark.parametrize("B, N", [(1, 5), (2, 3), (7, 1), (31, 129), (33, 38), (64, 33), (100, 515),
                                  (128, 1027), (129, 5), (255, 130), (257, 131),
                                  (300, 4), (513, 1000), (1000, 4096), (2049, 77), (4100, 256),
                                  (136, 12), (264, 2048), (512, 1000), (8192, 64)])
def test_edge_shapes_bit_exact(B, N):
    a = wl.make_reduce_input(B, N, seed=7 * B + N)
    np.testing.assert_array_equal(bits(gpu_reduce(a)), bits(oracle.reduce_axis0(a)))


@pytest.mark.parametrize("in_off, out_off", [(1, 0), (0, 1), (2, 3), (4, 4)])
def test_unaligned_pointers_take_the_scalar_path(in_off, out_off):
    a = wl.make_reduce_input(40, 1024, seed=3)
    got = gpu_reduce(a, out_offset=out_off, in_offset=in_off)
    np.testing.assert_array_equal(bits(got), bits(oracle.reduce_axis0(a)))


def test_empty_batch_writes_positive_zero():
    torch = torch_mod()
    out = torch.full((100,), float("nan"), device="cuda")
    cfc.reduce_axis0(torch.empty(0, 100, device="cuda"), out)
    assert np.all(bits(out.cpu().numpy()) == 0)


@pytest.mark.parametrize("name, col, expect", load_reduce_golden())
def test_golden_columns(name, col, expect):
    if col.size == 0:
        pytest.skip("empty batch covered above")
    a = np.repeat(col.reshape(-1, 1), 8, axis=1)     # 8 identical columns, float4 path
    got = gpu_reduce(a)
    assert np.all(bits(got) == bits(np.array([expect], np.float32))[0]), name


def test_integer_valued_exact():
    B, N = 1500, 4099
    b = np.arange(B)[:, None]
    j = np.arange(N)[None, :]
    a = (((7 * b + j) % 13) - 6).astype(np.float32)
    np.testing.assert_array_equal(gpu_reduce(a), a.astype(np.int64).sum(0).astype(np.float32))


def test_run_to_run_bit_identical():
    torch = torch_mod()
    a = dev(wl.make_reduce_input(1024, 40960, seed=11))
    ref = None
    for _ in range(10):
        out = torch.empty(40960, device="cuda")
        cfc.reduce_axis0(a, out)
        cur = bits(out.cpu().numpy())
        if ref is None:
            ref = cur
        else:
            np.testing.assert_array_equal(cur, ref)


MULTI_SHAPES = [(1024, 40960), (256, 40961), (32, 4096), (0, 100), (7, 1), (300, 131), (129, 5),
                (64, 1027), (1, 37), (2049, 77), (33, 4), (100, 515), (1031, 8)]


@pytest.mark.parametrize("repeat", [1, 4])          # 13 or 52 matrices (more than one launch's table)
def test_multi_matches_single_calls_bitwise(repeat):
    """reduce_axis0_multi over a mixed list (float4 and scalar configurations,
    every batch band, empty batch, ragged and unaligned rows) gives, for every
    matrix, the oracle's bits."""
    torch = torch_mod()
    shapes = MULTI_SHAPES * repeat
    mats, outs, refs = [], [], []
    for i, (B, N) in enumerate(shapes):
        a = wl.make_reduce_input(B, N, seed=97 * i + B)
        off = i % 3                                      # some inputs not 16-byte aligned
        flat = torch.full((off + B * N,), float("nan"), device="cuda")
        flat[off:] = dev(a.reshape(-1))
        mats.append(flat[off:].view(B, N))
        outs.append(torch.full((N,), float("nan"), device="cuda"))
        refs.append(oracle.reduce_axis0(a))
    cfc.reduce_axis0_multi(mats, outs)
    torch.cuda.synchronize()
    for i, (o, ref) in enumerate(zip(outs, refs)):
        np.testing.assert_array_equal(bits(o.cpu().numpy()), bits(ref), err_msg=f"matrix {i} {shapes[i]}")


def test_multi_empty_list_and_single_entry():
    torch = torch_mod()
    cfc.reduce_axis0_multi([], [])
    a = wl.make_reduce_input(256, 40960, seed=1)
    out = torch.empty(40960, device="cuda")
    cfc.reduce_axis0_multi([dev(a)], [out])
    np.testing.assert_array_equal(bits(out.cpu().numpy()), bits(oracle.reduce_axis0(a)))
