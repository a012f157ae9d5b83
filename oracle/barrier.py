"""Oracle: the N-rank notify/wait barrier and the builtin reveal.  TEST INFRASTRUCTURE ONLY.

Restated from the PyPTO page "Barrier: Signals Only" (sections The idea, Walkthrough, Edge
cases):

* Every rank owns one row of every peer's ``[N, 1]`` int32 signal window.  Notify adds 1
  (AtomicAdd) to row ``my_rank`` of each peer's window; wait blocks until row ``src`` of the
  rank's own window is >= the expected value (Ge), for every src other than itself.  A rank
  never notifies itself, so after one barrier rank r's column reads 1 everywhere but row r.
* Counters are monotonic: the gen-th use of one window waits for >= gen.
* The builtin reveal: each rank stages x into ``data``, passes a barrier that leaves no tally
  in the signal window, then reads the next rank's ``data``: y[r] = x[(r + 1) % N].
* Pitfall: a Set/Eq barrier on one shared cell lets later writes clobber earlier ones and can
  pass before every peer has arrived.
"""
from __future__ import annotations

from typing import List

import numpy as np


def handrolled(signal: np.ndarray, gen: int) -> np.ndarray:
    """One use of the hand-rolled barrier on windows ``signal[P, P]`` (rank, row); returns y.

    ``signal[q, i]`` is row i of rank q's window.  Mutates ``signal``; returns y[P, P] with
    y[r, i] = signal[r, i] read after rank r's waits have passed.
    """
    P = signal.shape[0]
    for r in range(P):                       # notify phase
        for peer in range(P):
            if peer != r:
                signal[peer, r] += 1
    y = np.zeros_like(signal)
    for r in range(P):                       # wait phase: sequentially every wait holds
        for src in range(P):
            if src != r and signal[r, src] < gen:
                raise RuntimeError(f"rank {r} would wait forever on row {src}")
        y[r] = signal[r]
    return y


def expected_column(P: int, r: int, gen: int = 1) -> np.ndarray:
    """Rank r's window after ``gen`` barriers: gen in every row but its own (0)."""
    col = np.full(P, gen, dtype=np.int32)
    col[r] = 0
    return col


def reveal(x: np.ndarray) -> np.ndarray:
    """Builtin reveal: stage x into data, barrier, then y[r] = data[(r + 1) % P]."""
    P = x.shape[0]
    data = x.copy()
    return np.stack([data[(r + 1) % P] for r in range(P)])


# --- the shared-cell pitfall (edge-case table), as scripted interleavings ----------------------
def shared_cell_set_eq(arrivals: List[int], P: int) -> bool:
    """Set/Eq on one shared cell: each arriving rank overwrites the cell with 1; a waiter passes
    when the cell equals 1.  Returns whether rank 0's wait passes after ``arrivals`` (the ranks
    that have arrived so far, in order)."""
    cell = 0
    for _ in arrivals:
        cell = 1                             # plain overwrite: earlier arrivals are lost
    return cell == 1


def shared_cell_add_ge(arrivals: List[int], P: int) -> bool:
    """AtomicAdd/Ge on one shared cell: the waiter passes once the cell is >= P."""
    cell = 0
    for _ in arrivals:
        cell += 1
    return cell >= P
