"""Helpers shared by the GPU parity tests: the oracle side of a workload (oracle/run.py) and
sampled byte offsets for full-size workloads."""
import numpy as np

from oracle.run import expected_bytes, make_plan as oracle_plan, run_round as oracle_round  # noqa: F401


def sample_offsets(w, n, seed, o=None):
    """Random byte offsets plus the first and last bytes of every region's first and last row."""
    rng = np.random.default_rng(seed)
    offs = [rng.integers(0, w.buf_bytes, n, dtype=np.int64)]
    if o is not None:
        ends = []
        for ch in o.chunks:
            for (off, rb, rows, pitch) in ch.regions:
                last = off + (rows - 1) * pitch + rb - 1
                ends += [off, off + rb - 1, last, last - rb + 1]
        offs.append(np.asarray(ends, dtype=np.int64))
    return np.unique(np.concatenate(offs))
