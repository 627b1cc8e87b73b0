"""Host-side pieces of bench.py that need no GPU: the packed buffers through
which the end-to-end step moves its inputs and gradients with one copy each
way, and the per-kernel traffic table's source hashes."""

import importlib.util
import os

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_packed_block_views_are_disjoint_aligned_and_round_trip(bench):
    specs = [("x", torch.bfloat16, (5, 3, 7)), ("b", torch.float32, (3, 11)),
             ("dt", torch.float32, (1,)), ("W", torch.float32, (3, 4, 9))]
    p = bench.packed_block(torch, specs, device="cpu")
    base = p.buf.data_ptr()
    spans = []
    for name, dt, shape in specs:
        v = p.views[name]
        assert v.dtype == dt and tuple(v.shape) == shape and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0                      # no two views overlap
    assert spans[-1][1] <= p.buf.numel()
    # writing every view and copying the block carries every tensor along
    rng = np.random.default_rng(0)
    for name, dt, shape in specs:
        p.views[name].copy_(torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dt))
    q = bench.packed_block(torch, specs, device="cpu")
    q.buf.copy_(p.buf)
    for name, _, _ in specs:
        assert torch.equal(q.views[name], p.views[name])


def test_traffic_table_names_known_kernels(bench):
    for (workload, name), (nbytes, digest) in bench.PROFILED_TRAFFIC.items():
        assert workload in ("smoke", "mid", "large") and nbytes > 0
        assert name in bench.KERNEL_FILES
        assert len(digest) == 16 and len(bench.kernel_source_hash(name)) == 16
