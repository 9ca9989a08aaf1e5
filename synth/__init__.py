"""Seeded synthetic inputs shared by the oracle-side tests, the GPU tests and the bench.

This package draws random numbers and builds allowed-key sets; it holds none of the
attention arithmetic (no scores, no softmax, no gradients).
"""
from .inputs import (  # noqa: F401
    CONFIGS,
    Workload,
    bitmap_mask,
    draw_head,
    draw_tensor,
    pack_bitmap,
    random_allowed,
    round_to_dtype,
    workload,
)
