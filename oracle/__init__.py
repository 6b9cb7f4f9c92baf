"""CPU oracle for the chunk-centric fused AllGather-GEMM, GEMM-ReduceScatter,
GEMM-AllReduce and GEMM-AllToAll.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
anything here: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` (and its ``--impl reference`` arm) may use it.

The oracle is plain and slow on purpose.  It computes in float64 from the exact
values of the bf16 inputs and shares no code with the CUDA path:

* ``reference``  - concat-then-matmul (AllGather-GEMM) and
  per-rank-partial-sum-then-row-scatter (GEMM-ReduceScatter), full and sampled;
* ``plan``       - the chunk map, the rank-aware tile orders (gather and
  scatter modes of the distributed swizzle), the chunk transfer order and the
  per-unit arrival counts, each written straight from its definition (sorting
  by key), with no closed forms.

Every function is pinned by the ``-m "not gpu"`` tests against brute force,
closed forms, special cases and the worked order of the DITRON page (Fig. 3).
"""
from . import plan, reference  # noqa: F401
