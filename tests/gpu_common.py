"""Helpers shared by the GPU parity tests: the oracle side of a workload (oracle/run.py), the
oracle's whole expected buffer (oracle/cfill.py), and sampled byte offsets."""
import numpy as np

from oracle import cfill
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


def expected_on_device(w, rnd):
    """The oracle's closed form of every buffer after round rnd (computed on the host by the C
    oracle), moved to the device so that whole buffers can be compared there."""
    import torch
    return torch.from_numpy(cfill.expected_buffer(w, rnd)).cuda()


def assert_buffers_equal(bufs, want, what):
    """Every byte of every buffer equals the oracle's; on a mismatch name the first bad byte."""
    import torch
    for q, b in enumerate(bufs):
        if torch.equal(b, want):
            continue
        bad = (b != want).nonzero()
        first = int(bad[0, 0])
        raise AssertionError(f"{what}: buffer {q} differs from the oracle at {bad.shape[0]} byte(s), "
                             f"first at offset {first} (got {int(b[first])}, want {int(want[first])})")
