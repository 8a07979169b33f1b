"""CPU oracle for the swizzled-GEMM hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct restatements of what the three source pages
define, written independently of the CUDA library (no shared code, headers,
tables or helpers; neither side imports the other):

* ``tile_order``  -- program-id -> output-tile maps (row/col-major, grouped 2D
  panel, Morton, XOR, serpentine), the cluster-persistent work distribution and
  the cluster-tile -> CTA-tile split.
* ``l2_model``    -- the byte-granular LRU L2 hit-rate model and the Spearman
  rank correlation used to compare it with measured throughput.
* ``smem_bank``   -- shared-memory address functions (padding, XOR swizzles,
  TMA 128B swizzle, CuTe-style Swizzle<B,M,S>, Triton vec/perPhase/maxPhase)
  and a per-warp bank-conflict counter.
* ``ref``         -- FP64 GEMM and 32-bit transpose, in plain C (gemm_ref.c),
  loaded with ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or execute anything in
this package.  The product path never routes through it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values the pages print, closed forms, invariants or brute force --
except the GPU-measured L2 hit rate versus the L2 model, which the first page
itself calls directional only (parity unpinned).
"""
