"""CPU oracle for the triggered-plan all-gather.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU restatement of what the triggered-plan hot path computes:
the schedule builders, the gate and round semantics, the in-place all-gather result, the N-rank
notify/wait barrier and the GEMM producer's product.  It is written from the public
descriptions ("Triggered Plans" in the Iris docs, "Triggered SDMA Plans" = ROCm/iris pull 573,
and the PyPTO page "Barrier: Signals Only") and shares no code with the CUDA library in
``device_triggered_transfers_gb300``: neither imports the other.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it; the product
path never routes through it.

Modules and what pins each (see the test files named):

* ``hashfill``  synthetic producer values.  The pages fix no formula: the hash composition is
  builder-defined.  fmix32 is pinned by published MurmurHash3 vectors, the bf16 rounding by
  torch's conversion, the uniform mapping by closed form (tests/test_oracle_hash.py).  The salt
  composition itself has no pin beyond its definition: "parity unpinned" for that part.
* ``cfill``     the same values from a plain-C restatement (``fill.c``, compiled with gcc), so
  full-size buffers can be compared byte for byte.  Pinned by the same vectors and closed forms
  as ``hashfill`` and checked element by element against it (tests/test_oracle_hash.py).
* ``schedule``  whole / chunks / tile_chunks builders, the step-to-tile orders, the global
  chunk numbering and plan validation.  Pinned by golden counts, the 1 GiB split, coverage by
  brute-force ownership maps and the order special cases (tests/test_oracle_schedule.py).
  The GROUP_M grouped order is a reading (the pages elide its body): pinned only through its
  special cases (GROUP_M=1 is row-major, GROUP_M>=tiles_m is column-major) and bijectivity.
* ``plan``      the sequential round model: marks, gates, per-peer queues, wait, next_round,
  close.  Pinned by the closed-form all-gather result, gate invariants after R rounds and an
  exhaustive interleaving check (tests/test_oracle_plan.py).
* ``threaded``  the same protocol with CPU threads as ranks (tests/test_oracle_threaded.py).
* ``barrier``   hand-rolled notify/wait barrier and the builtin reveal, plus the Set/Eq
  shared-cell pitfall.  Pinned by the page's golden values (tests/golden/barrier_p*.txt).
* ``gemm``      fp64 product of the bf16 operands and the relative Frobenius error.  Pinned by
  brute force on tiny inputs and closed forms (tests/test_oracle_barrier_gemm.py).
* ``allreduce`` the two-shot all-reduce ("Triggered Plans", Not supported yet, names it): the
  sum in f32 in rank order, rounded once (a reading: the pages fix no precision), and the
  protocol of a reduce-scatter plan, the reduce step and an all-gather plan on the ``plan``
  model.  Pinned by hand-worked sums (tests/golden/allreduce_sums.txt), closed forms, the f32
  summation error bound against the exact sum, a brute-force bf16 rounding check and the
  protocol against the definition (tests/test_oracle_allreduce.py).
"""
from . import hashfill, schedule, plan, barrier, gemm, allreduce  # noqa: F401
