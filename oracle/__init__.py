"""CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it and
it never imports the CUDA library.  See ``cfc_oracle`` for the definitions
it follows and the rounding points it mirrors.
"""
from .cfc_oracle import (  # noqa: F401
    FP32, TF32, BF16, round_bf16, round_tf32, cell_forward, forward, backward,
    per_sample_length, unpack_per_sample, reduce_axis0,
)
