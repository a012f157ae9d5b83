"""Oracle: the two-shot all-reduce built from two triggered plans.  TEST INFRASTRUCTURE ONLY.

"Triggered Plans" (Iris docs), section Not supported yet, names two-shot all-reduce among what
other destinations (a copy landing at another offset or buffer, a chunk going to only some
peers) make possible, and says nothing more about it.  The reading taken here is the plain one:

* All-reduce: every rank ends with y = x_0 + x_1 + ... + x_{P-1}, element by element, over the
  P ranks' vectors of M = P * Mb rows of ``cols`` elements (bf16 or f32), rows ``pitch`` bytes
  apart at the start of each rank's buffer.
* Precision (the pages fix none): the sum is taken in f32, adding the ranks' values in rank
  order 0, 1, ..., P-1 with one IEEE round-to-nearest-even after every add, then rounded once to
  the element type (bf16: nearest even; f32: as it is).  A fixed order makes the result one
  number, so the device's result can be compared bit for bit.
* Two shots: a reduce-scatter, then an all-gather.  Rank b owns block b, rows [b*Mb, (b+1)*Mb).
  Shot one: every rank s sends its partial of block b to rank b, into slot s of b's staging
  area (slot s holds Mb rows at ``slot_off + s*Mb*pitch``, in b's own buffer after the vector
  or in a separate staging buffer); rank b adds its own partial and the P-1 slots in rank order
  and writes the sum over its own block.  Shot two: rank b sends its block to every other rank,
  at the same rows.
* Each block is cut into J chunks of Mb / J rows, so the shots pipeline chunk by chunk:
  reduce-scatter chunk (s, b, j) lands in slot s at rank b; group (b, j) holds the P chunks
  (s, b, j), s = 0..P-1 -- at rank b its own one counts when marked, the others when they
  arrive -- so one group wait at rank b says every part of (b, j) is there; the reduce then
  marks all-gather chunk (b, j).
* Chunk numbering: rank s's reduce-scatter chunks are (b, j) in the order b*J + j (row order of
  its vector); rank b's all-gather chunks are j = 0..J-1.  Group (b, j) is group b*J + j.
* Reduce-scatter, the other operation the same bullet names, is the first shot alone: rank b
  ends with the sum over its own block b; its other rows keep its own partial, and no
  all-gather plan exists (``gather=False``).
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from . import hashfill as H
from . import plan as OP
from . import schedule as S

ELEM_BYTES = {"bf16": 2, "f32": 4}
STORAGE = {"bf16": np.uint16, "f32": np.float32}


# -- the definition ------------------------------------------------------------------------
def to_f32(dtype: str, x: np.ndarray) -> np.ndarray:
    """Storage values (bf16 bits or float32) as float32 (exact for both)."""
    if dtype == "bf16":
        return H.bf16_bits_to_f32(x)
    return np.asarray(x, dtype=np.float32)


def from_f32(dtype: str, x: np.ndarray) -> np.ndarray:
    """float32 to the storage type: bf16 by round to nearest even, f32 as it is."""
    if dtype == "bf16":
        return H.f32_to_bf16_bits(x)
    return np.asarray(x, dtype=np.float32)


def allreduce(dtype: str, parts: Sequence[np.ndarray]) -> np.ndarray:
    """y = x_0 + ... + x_{P-1} in f32, in rank order, rounded once to ``dtype`` (storage values
    in, storage values out)."""
    acc = to_f32(dtype, parts[0]).copy()
    for x in parts[1:]:
        acc = (acc + to_f32(dtype, x)).astype(np.float32)   # float32 + float32: one IEEE rounding
    return from_f32(dtype, acc)


def exact_sum(dtype: str, parts: Sequence[np.ndarray]) -> np.ndarray:
    """The same sum in float64, without the f32 roundings (exact for up to 8 bf16 values whose
    exponents lie within 40 of each other); the tests' reference for the error bound."""
    return sum(to_f32(dtype, x).astype(np.float64) for x in parts)


# -- the two plans ---------------------------------------------------------------------------
def layout(P: int, Mb: int, cols: int, dtype: str, pitch: Optional[int] = None, separate: bool = False):
    """Byte sizes of the two-shot layout: (row_bytes, pitch, buf_bytes, slot_off, staging_bytes).
    In place the P slots follow the vector in each rank's buffer; with separate staging buffers
    they start at byte 0 of those."""
    rb = cols * ELEM_BYTES[dtype]
    pitch = pitch or rb
    M = P * Mb
    if separate:
        return rb, pitch, M * pitch, 0, P * Mb * pitch
    return rb, pitch, 2 * M * pitch, M * pitch, 0


def _rows_region(off: int, rb: int, rows: int, pitch: int):
    return (off, rb, rows, pitch) if rows > 1 else (off, rb, 1, rb)


def reduce_scatter_schedules(P: int, Mb: int, J: int, rb: int, pitch: int, slot_off: int) -> List[S.Schedule]:
    """Rank s's chunk (b, j): rows [b*Mb + j*Mj, +Mj) of its vector, to rank b only, landing in
    slot s of b's staging area at the same rows of the block (Mj = Mb / J)."""
    Mj = Mb // J
    out = []
    for s in range(P):
        chunks = []
        for b in range(P):
            for j in range(J):
                src = _rows_region((b * Mb + j * Mj) * pitch, rb, Mj, pitch)
                dst = (slot_off + (s * Mb + j * Mj) * pitch, src[3])
                chunks.append(S.Chunk([src], 1, dests=[dst], peers=1 << b))
        out.append(S.Schedule(chunks))
    return out


def reduce_groups(P: int, J: int) -> List[List[int]]:
    """Group (b, j) = b*J + j: the global ids of chunk (s, b, j) for s = 0..P-1 (rank s's chunks
    are numbered after the P*J of each lower rank)."""
    return [[s * P * J + b * J + j for s in range(P)] for b in range(P) for j in range(J)]


def allgather_schedules(P: int, Mb: int, J: int, rb: int, pitch: int) -> List[S.Schedule]:
    """Rank b's chunk j: rows [b*Mb + j*Mj, +Mj), to every other rank at the same rows."""
    return [S.chunks(b * Mb * pitch, Mb, rb, pitch, J) for b in range(P)]


class TwoShot:
    """The two plans over P byte buffers (and staging buffers), with the reduce step between
    them, driven through the oracle's plan model one round at a time."""

    def __init__(self, P: int, Mb: int, cols: int, dtype: str, J: int, pitch: Optional[int] = None,
                 separate: bool = False, initial_round: int = 1, gather: bool = True):
        if Mb % J:
            raise ValueError("J must divide the block rows")
        self.P, self.Mb, self.cols, self.dtype, self.J = P, Mb, cols, dtype, J
        self.Mj = Mb // J
        self.rb, self.pitch, self.buf_bytes, self.slot_off, self.staging_bytes = \
            layout(P, Mb, cols, dtype, pitch, separate)
        self.bufs = [np.zeros(self.buf_bytes, dtype=np.uint8) for _ in range(P)]
        self.staging = [np.zeros(self.staging_bytes, dtype=np.uint8) for _ in range(P)] if separate else None
        self.rs = OP.Plan(self.bufs, reduce_scatter_schedules(P, Mb, J, self.rb, self.pitch, self.slot_off),
                          allgather=False, dst_bufs=self.staging, initial_round=initial_round)
        self.rs.define_groups(reduce_groups(P, J))
        self.gather = gather
        self.ag = OP.Plan(self.bufs, allgather_schedules(P, Mb, J, self.rb, self.pitch),
                          allgather=False, initial_round=initial_round) if gather else None

    # rows of a byte buffer as storage values
    def _rows(self, buf: np.ndarray, off: int, rows: int) -> np.ndarray:
        t = STORAGE[self.dtype]
        out = np.empty((rows, self.cols), dtype=t)
        for i in range(rows):
            a = off + i * self.pitch
            out[i] = buf[a:a + self.rb].view(t)
        return out

    def _put_rows(self, buf: np.ndarray, off: int, vals: np.ndarray) -> None:
        for i in range(vals.shape[0]):
            a = off + i * self.pitch
            buf[a:a + self.rb] = np.ascontiguousarray(vals[i]).view(np.uint8)

    def stage(self, b: int) -> np.ndarray:
        return self.staging[b] if self.staging is not None else self.bufs[b]

    def reduce_chunk(self, b: int, j: int) -> None:
        """The reduce step for (b, j): rank b's own partial rows and slots 0..P-1 (its own slot
        is never written: its own partial stands in for it), added in rank order."""
        g = b * self.J + j
        if not self.rs.group_ready(b, g):
            raise OP.StateError(f"reduce of ({b}, {j}) before its group is complete")
        row0 = b * self.Mb + j * self.Mj
        parts = []
        for s in range(self.P):
            if s == b:
                parts.append(self._rows(self.bufs[b], row0 * self.pitch, self.Mj))
            else:
                parts.append(self._rows(self.stage(b), self.slot_off + (s * self.Mb + j * self.Mj) * self.pitch, self.Mj))
        self._put_rows(self.bufs[b], row0 * self.pitch, allreduce(self.dtype, parts))
        if self.gather:
            self.ag.mark_ready(b, self.ag.first[b] + j)

    def round(self, partials: Sequence[np.ndarray]) -> int:
        """One round: every rank's partial vector ([M, cols] storage values) written and its
        reduce-scatter chunks marked, the copies, the reduce of every (b, j), the all-gather
        copies, both waits, both next_rounds.  Returns the round."""
        R = self.rs.start()
        if self.gather and self.ag.start() != R:
            raise OP.StateError("the two plans are in different rounds")
        for s in range(self.P):
            self._put_rows(self.bufs[s], 0, np.asarray(partials[s]))
            for c in self.rs.chunks_of(s):
                self.rs.mark_ready(s, c)
        self.rs.copier_progress()
        for b in range(self.P):
            for j in range(self.J):
                self.reduce_chunk(b, j)
        if self.gather:
            self.ag.copier_progress()
        for pl in (self.rs, self.ag) if self.gather else (self.rs,):
            st = pl.wait()
            if st[0] != OP.OK:
                raise OP.StateError(f"round {R} failed: {st}")
            pl.next_round()
        return R

    def result(self, r: int) -> np.ndarray:
        """Rank r's vector rows as storage values."""
        return self._rows(self.bufs[r], 0, self.P * self.Mb)


def reduce_scatter(dtype: str, parts: Sequence[np.ndarray], P: int, Mb: int) -> List[np.ndarray]:
    """Each rank's vector after a reduce-scatter: block b of rank b is the sum (as ``allreduce``)
    of every rank's block b; its other blocks are its own partial as it was."""
    y = allreduce(dtype, parts)
    out = []
    for b in range(P):
        v = np.array(parts[b], copy=True)
        v[b * Mb:(b + 1) * Mb] = y[b * Mb:(b + 1) * Mb]
        out.append(v)
    return out


def hashed_partials(dtype: str, seed: int, P: int, M: int, cols: int, rnd: int) -> List[np.ndarray]:
    """The partial vectors of the fill producer: rank r's [M, cols] in round rnd (the hashed
    uniform values of ``hashfill``)."""
    return [H.fill_slice(dtype, seed, r, rnd, M, cols) for r in range(P)]
