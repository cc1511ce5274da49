"""CPU oracle for the FP32 SGEMM path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import or run anything here.  The GPU
library (``dense_fp32_matrix_04_gb300``) never imports, links or calls it, and
the two share no code: the only module both sides use is the seeded input
generator ``gen``, which holds none of the product's arithmetic.

Contents
--------
* ``ref_gemm``: plain C triple loop with FP64 accumulation (the definition of
  C = A * B written out), plus the absolute-value sum used by the tolerance.
* ``tilesim``: counting simulator of the pages' naive, tiled and register-tiled
  kernels (global and shared reads, multiply-adds) and the 32-bank model.
* ``tolerance``: the elementwise acceptance test for an FP32 result.

Pins (what the oracle is checked against, in ``tests/test_oracle_*.py``):
exact small-integer and identity products, brute-force exact sums at 6 x 6 x 9,
an independent FP64 library product, closed forms, and every figure the pages
print for their worked examples (``tests/golden/``).  One count has no printed
value: register reads (two per multiply-add) -- parity unpinned.
"""
