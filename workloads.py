"""Synthetic workloads for the triggered all-gather: shapes, seeds and seeded input generators.

This module holds the recipes only (sizes, schedule kinds, seeds) and the seeded random
generators for inputs that are data rather than produced values (GEMM operands, barrier
payloads).  It holds none of the method's arithmetic: the producer's hashed values, the
schedules, the gate protocol and the copies are implemented separately by the CPU oracle
(``oracle/``) and by the CUDA library, and both read their workload description from here.

The five workloads mirror the functional tests described in "Triggered SDMA Plans" (ROCm/iris
pull 573, section Testing) and the Iris "Triggered Plans" page (section Model): 1D chunks, 2D
tiles with clipped edges, 8 writers on one 4 MiB gate for 10 rounds, a broadcast split into
1 GiB copies, and a GEMM producer.  The N-rank barrier follows the PyPTO page "Barrier:
Signals Only".
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BASE_SEED = 20261202

BF16, F32, U8 = "bf16", "f32", "u8"
ELEM_BYTES = {BF16: 2, F32: 4, U8: 1}


@dataclass(frozen=True)
class Workload:
    """One all-gather (or broadcast) workload over P virtual ranks in one GPU.

    Every virtual rank owns a buffer of ``P*M`` rows (all-gather) or ``M`` rows (broadcast)
    by ``N`` elements of ``dtype``.  Rank r's slice is rows ``[r*M, (r+1)*M)`` of its own
    buffer (all-gather) or the whole buffer of the single sender (broadcast).
    ``kind`` is the schedule builder: ``whole`` (``num_programs`` writers on one chunk),
    ``chunks`` (``num_chunks`` row blocks, one writer each) or ``tile_chunks``
    (``BM`` x ``BN`` tiles, ``tiles_per_chunk`` consecutive producer steps per chunk,
    ``group_m`` > 0 selects the grouped step-to-tile order).
    """
    name: str
    P: int
    M: int
    N: int
    dtype: str
    kind: str
    rounds: int
    seed: int
    num_programs: int = 1
    num_chunks: int = 1
    BM: int = 0
    BN: int = 0
    tiles_per_chunk: int = 0
    group_m: int = 0
    broadcast: bool = False
    K: int = 0                      # GEMM producer only: inner dimension

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def row_bytes(self) -> int:
        return self.N * self.elem_bytes

    @property
    def buf_rows(self) -> int:
        return self.M if self.broadcast else self.P * self.M

    @property
    def buf_bytes(self) -> int:
        return self.buf_rows * self.row_bytes

    @property
    def slice_bytes(self) -> int:
        return self.M * self.row_bytes

    def senders(self):
        return [0] if self.broadcast else list(range(self.P))

    def slice_offset(self, r: int) -> int:
        return 0 if self.broadcast else r * self.slice_bytes

    def delivered_bytes_per_round(self) -> int:
        """Bytes landed in peers per round: every sender's slice to P-1 peers."""
        return len(self.senders()) * self.slice_bytes * (self.P - 1)

    def algorithmic_bytes_per_round(self) -> int:
        """HBM bytes a read-once, fan-out copier must move per round (read + writes)."""
        return len(self.senders()) * self.slice_bytes * self.P


# The five measured workloads (seed = BASE_SEED + index).
C1 = Workload("c1_whole_p2", P=2, M=256, N=256, dtype=BF16, kind="whole", rounds=3,
              seed=BASE_SEED + 1, num_programs=1)
C2 = Workload("c2_chunks_p4", P=4, M=4096, N=4096, dtype=BF16, kind="chunks", rounds=10,
              seed=BASE_SEED + 2, num_chunks=8)
C3 = Workload("c3_tiles_p8", P=8, M=8000, N=8064, dtype=BF16, kind="tile_chunks", rounds=10,
              seed=BASE_SEED + 3, BM=128, BN=128, num_programs=148, tiles_per_chunk=148,
              group_m=8)
C4A = Workload("c4a_writers8_p8", P=8, M=1024, N=1024, dtype=F32, kind="whole", rounds=10,
               seed=BASE_SEED + 4, num_programs=8)
# 2.5 GiB uint8 broadcast from rank 0: 2560 rows of 1 MiB.
C4B = Workload("c4b_bcast_p8", P=8, M=2560, N=1 << 20, dtype=U8, kind="whole", rounds=1,
               seed=BASE_SEED + 4, num_programs=152, broadcast=True)
C5 = Workload("c5_gemm_p4", P=4, M=2048, N=4096, dtype=BF16, kind="tile_chunks", rounds=5,
              seed=BASE_SEED + 5, BM=128, BN=128, num_programs=148, tiles_per_chunk=148,
              group_m=0, K=4096)

CONFIGS = {w.name: w for w in (C1, C2, C3, C4A, C4B, C5)}

# The two-shot all-reduce ("Triggered Plans", Not supported yet, names it): P = 4 ranks whose
# vectors are bf16 [16384, 4096] (128 MiB each, the size of the 4-rank chunked all-gather), so
# each rank reduces a 4096-row block, cut into 4 sub-blocks of 1024 rows (8 MiB: each sub-block
# is one reduce-scatter chunk, and a copier CTA drains its stores once per chunk, so 4 MiB
# sub-blocks made rounds ~7 % longer); the producer writes the hashed values of every rank's
# vector, a group of 38 CTAs per rank.
ALLREDUCE = dict(name="allreduce_p4", P=4, block_rows=4096, cols=4096, sub_blocks=4, dtype=BF16,
                 seed=BASE_SEED + 6, fill_group=38)

BARRIER_P = 8
BARRIER_SIZE = 256
BARRIER_SEED = BASE_SEED + 4


def barrier_payload(P: int = BARRIER_P, size: int = BARRIER_SIZE,
                    seed: int = BARRIER_SEED) -> np.ndarray:
    """Seeded int32 payload x[r, :] staged by each virtual rank before the reveal barrier."""
    rng = np.random.default_rng(seed)
    return rng.integers(-(1 << 31), 1 << 31, size=(P, size), dtype=np.int64).astype(np.int32)


def gemm_inputs(P: int, M: int, N: int, K: int, seed: int):
    """Seeded GEMM operands: A_r [M, K] per rank and a shared B [K, N] (stored as [N, K]).

    Entries are N(0, 1)/sqrt(K), rounded to bf16.  Returned as torch bf16 CPU tensors:
    ``A`` of shape [P, M, K] (row-major, K contiguous) and ``Bt`` of shape [N, K]
    (B transposed, K contiguous), the K-major layout both operands use on the device.
    """
    import torch
    g = torch.Generator().manual_seed(seed)
    scale = 1.0 / float(np.sqrt(K))
    A = (torch.randn(P, M, K, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)
    Bt = (torch.randn(N, K, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)
    return A, Bt


def small(w: Workload, **over) -> Workload:
    """A copy of ``w`` with some fields replaced (for parity cases the oracle finishes fast)."""
    d = dict(w.__dict__)
    d.update(over)
    return Workload(**d)
