"""Host-side data-parallel logic on CPU: batch slicing, packed gradient views and
the cross-rank gradient exchange (all_gather in rank order + fixed-order
reduction) with world_size 2 over gloo.  Every rank computes its slice's
gradient with the oracle and exchanges it; the exchanged sum must be
bit-identical on both ranks, equal the oracle's reduction of the gathered
rows, and match the full-batch gradient (the reduced gradient is the sum of
the per-sample gradients, whatever the split)."""

import os
import socket

import numpy as np
import pytest

import oracle
from recurrent_cell_gb300 import dp
from recurrent_cell_gb300 import workloads as wl


@pytest.mark.parametrize("B, world", [(7, 2), (8, 2), (5, 3), (2, 4), (0, 2), (1031, 8)])
def test_shard_bounds_partition_the_batch(B, world):
    bounds = [dp.shard_bounds(B, r, world) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == B
    for (s0, e0), (s1, e1) in zip(bounds, bounds[1:]):
        assert e0 == s1
    sizes = [e - s for s, e in bounds]
    assert max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)


def test_shard_bounds_rejects_bad_rank():
    with pytest.raises(ValueError):
        dp.shard_bounds(4, 2, 2)
    with pytest.raises(ValueError):
        dp.shard_bounds(4, 0, 0)


def test_gradient_views_follow_per_sample_packing():
    import torch
    n_in, H = 16, 32
    N = dp.packed_length(n_in, H)
    assert N == oracle.per_sample_length(n_in, H)
    flat = torch.arange(N, dtype=torch.float32)
    gWi, gWr, gb = dp.gradient_views(flat, n_in, H)
    ref = oracle.unpack_per_sample(flat.numpy(), n_in, H)
    for got, want in zip((gWi, gWr, gb), ref):
        np.testing.assert_array_equal(got.numpy(), want)
    assert gWi.data_ptr() == flat.data_ptr()          # views, not copies
    with pytest.raises(ValueError):
        dp.gradient_views(flat[:-1], n_in, H)
    with pytest.raises(ValueError):
        dp.gradient_views(torch.zeros(dp.packed_length(3, 5)), 3, 5)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


W = wl.Workload("dp_gloo_B7_K5_8x12_fp32", B=7, K=5, n_in=8, n_hid=12, dt_per_sample=True)


def _local_gradient(inp, lo, hi):
    """The slice's packed float32 gradient as the library's scratch path forms it:
    per-sample rows reduced in the canonical order."""
    sl = {k: inp[k][lo:hi] for k in ("x", "h0", "dt", "y")}
    out = oracle.backward(sl["x"], sl["h0"], inp["W_in"], inp["W_rec"], inp["b"], sl["dt"],
                          y=sl["y"], per_sample=True)
    return oracle.reduce_axis0(out["per_sample"].astype(np.float32))


def _rank_main(rank, world, port, outdir):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = wl.make_inputs(W)
        lo, hi = dp.shard_bounds(W.B, rank, world)
        local = torch.from_numpy(_local_gradient(inp, lo, hi))
        out = torch.full((W.N,), float("nan"))

        def reducer(gathered, o):
            o.copy_(torch.from_numpy(oracle.reduce_axis0(gathered.numpy())))

        dp.reduce_gradients(local, out, reducer=reducer)
        np.save(os.path.join(outdir, f"rank{rank}.npy"), out.numpy())
    finally:
        dist.destroy_process_group()


def test_gradient_exchange_world_size_2(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [np.load(tmp_path / f"rank{r}.npy") for r in range(world)]
    np.testing.assert_array_equal(got[0].view(np.uint32), got[1].view(np.uint32))

    inp = wl.make_inputs(W)
    rows = np.stack([_local_gradient(inp, *dp.shard_bounds(W.B, r, world)) for r in range(world)])
    np.testing.assert_array_equal(got[0].view(np.uint32), oracle.reduce_axis0(rows).view(np.uint32))

    full = oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"],
                           y=inp["y"], per_sample=False)
    want = np.concatenate([full["grad_W_in"].ravel(), full["grad_W_rec"].ravel(),
                           full["grad_b"].ravel()])
    np.testing.assert_allclose(got[0], want, rtol=1e-4, atol=1e-5)
