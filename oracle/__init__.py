"""CPU oracle for exact tiled softmax attention — TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 numpy restatements of what the attention path computes, written from
the pages on exact IO-aware attention:

* ``attention``  — the dense definition (materialises the score and probability matrices).
* ``tiled``      — the block-by-block summary/merge forward and the per-element reverse
                   procedure of "Exact tiled attention and memory-aware differentiation".
* ``masks``      — allowed-key sets: none, causal, and the packed bitmap the library reads.
* ``io_model``   — a global-memory byte counter for the unfused and fused kernels of the
                   "Night School: fused attention" lab.
* ``fp8``        — E4M3 rounding and the FP8 forward's exact reference with its error bound.
* ``dropout``    — the dropout extension with a replayed realised mask (Philox4x32-10 mask,
                   forward and reverse pass with the mask held fixed).

Only the test suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import
this package.  The GPU library never does, and this package imports nothing from it.
Every function here is pinned by ``-m "not gpu"`` tests against worked examples, closed
forms, invariants or brute force; none is marked "parity unpinned".
"""
from . import attention, dropout, fp8, io_model, masks, tiled  # noqa: F401
