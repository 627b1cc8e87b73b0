"""Data-parallel K-loop step over several ranks (one GPU per rank).

Samples are independent through the whole K loop, so the batch is split into
contiguous slices, one per rank, and every rank runs the forward and backward
of its slice with the C ABI.  The one exchange of the method is the parameter
gradient: each rank's gradient, packed as one [N] vector
[grad_W_in | grad_W_rec | grad_b] (N = 3 (n_in + n_hid + 1) n_hid, the packing
of the per-sample rows), is gathered into [G, N] in rank order and summed with
reduce_axis0.  The sum is deterministic and bit-identical on every rank; it is
the canonical fixed-order reduction, applied across ranks instead of samples.

This module holds plumbing only (slicing, views, the collective); the
arithmetic is the library's reduce_axis0 (or, in host-side tests, any reducer
with the same semantics passed in).
"""

from __future__ import annotations


def shard_bounds(B: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of rank's contiguous slice of B samples (sizes differ by
    at most one, lower ranks first)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def packed_length(n_in: int, n_hid: int) -> int:
    return 3 * (n_in + n_hid + 1) * n_hid


def gradient_views(flat, n_in: int, n_hid: int):
    """(grad_W_in [3,H,n_in], grad_W_rec [3,H,H], grad_b [3,H]) as views of the
    packed [N] vector ``flat``, in the per-sample row order."""
    H = n_hid
    a = 3 * H * n_in
    b = a + 3 * H * H
    if flat.numel() != b + 3 * H:
        raise ValueError(f"packed gradient has {flat.numel()} elements, expected {b + 3 * H}")
    if a % 4 or b % 4:
        # The library wants 16-byte aligned gradient buffers; the views start at
        # 4a and 4b bytes into the vector.
        raise ValueError(f"n_hid*n_in and n_hid*(n_in+n_hid) must be multiples of 4 for packed "
                         f"views (n_in={n_in}, n_hid={n_hid})")
    return flat[:a].view(3, H, n_in), flat[a:b].view(3, H, H), flat[b:].view(3, H)


def reduce_gradients(local, out, group=None, reducer=None, gathered=None):
    """out[N] = sum over ranks of every rank's ``local`` [N] gradient, in rank
    order through ``reducer`` (default: the library's reduce_axis0 on the
    device).  ``gathered`` is an optional preallocated [world, N] buffer.
    Collective: every rank of ``group`` must call it."""
    import torch
    import torch.distributed as dist
    if reducer is None:
        from . import reduce_axis0 as reducer
    world = dist.get_world_size(group)
    n = local.numel()
    if gathered is None:
        gathered = torch.empty((world, n), dtype=local.dtype, device=local.device)
    elif tuple(gathered.shape) != (world, n):
        raise ValueError(f"gathered buffer {tuple(gathered.shape)}, expected {(world, n)}")
    dist.all_gather([gathered[i] for i in range(world)], local.reshape(n).contiguous(), group=group)
    reducer(gathered, out)
    return out
