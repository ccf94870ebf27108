"""Oracles for the fused-epilogue GEMM and its layout algebra.  TEST INFRASTRUCTURE ONLY.

This package is the slow, plain CPU statement of what the CUDA path computes.
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import it; the product path never does, and it shares no code with
the CUDA sources.

* ``gemm_oracle.c`` / ``gemm_ref.py``: fp64 GEMM with the fused epilogue and
  round-to-nearest-even output rounding, one row at a time (C, OpenMP).
* ``layout_ref.py``: the shape:stride layout algebra (evaluation, coalesce,
  composition, complement, logical/zipped divide, local tile/partition).

Both are pinned in ``tests/test_oracle_*.py`` against brute force, closed
forms and the worked examples printed on the pages (``tests/golden/``).
"""
