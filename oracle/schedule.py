"""Oracle: schedule builders, step-to-tile orders, global chunk numbering, plan validation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources ("Triggered Plans", Iris docs, section Model and section Requirements and limits;
"Triggered SDMA Plans", ROCm/iris pull 573, section API):

* A region is one copy: a byte range, or a 2D sub-window (rows of a strided tensor), written at
  the same offset in every peer's buffer.  Linear copies move at most 1 GiB, so builders split
  longer byte ranges; 1 GiB is read as 2**30 bytes.
* A chunk is an ordered group of regions behind one gate, with ``writers`` marks per round.
* ``whole()``: one chunk, marked once per program at the end (writers = number of programs).
* ``chunks()``: row blocks completed in order, one writer each.  Block size is read as
  ceil(M / n) rows, the last block shorter.
* ``tile_chunks()``: consecutive producer steps; step s stores tile ``order(s)``; one 2D region
  per tile, clipped at the slice edges; chunk k holds steps [k*T, (k+1)*T).  Writers = the
  number of steps in the chunk (the producer marks once per tile).
* The producer marks ``first_chunk + step // num_programs``: chunk ids are global, each rank's
  chunks numbered after those of all lower ranks.
* ``prepare_all_gather`` checks that each rank's schedule stays inside its own rows; a plan
  rejects two ranks that send the same bytes.

A region is the tuple ``(offset, row_bytes, rows, pitch)``; a byte range has ``rows == 1`` and
``pitch == row_bytes``.  Offsets are relative to the start of the buffer.

Other destinations ("Triggered Plans", Not supported yet: a copy cannot change offset, pitch or
buffer, and a chunk cannot go to only some peers; reduce-scatter and two-shot all-reduce need
both).  Reading: a chunk may name, per region, a destination ``(offset, pitch)`` -- the same
rows of the same width land there instead of at the source's offset -- and a set of receiving
peers (a bit mask; none given: every other rank).  The destination is the receiving rank's
buffer, or its destination buffer when the plan has separate ones (a staging buffer).  The
checks that keep ranks from sending the same bytes extend to destinations: no two copies land
on the same bytes of one buffer, and, in place, no copy lands on bytes the receiving rank
itself sends.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

GiB = 1 << 30
LINEAR_MAX = GiB

Region = Tuple[int, int, int, int]   # (offset, row_bytes, rows, pitch)


@dataclass
class Chunk:
    regions: List[Region]
    writers: int
    dests: Optional[List[Tuple[int, int]]] = None   # per region (dst offset, dst pitch); None: same
    peers: Optional[int] = None                     # receiving ranks as a bit mask; None: all

    @property
    def nbytes(self) -> int:
        return sum(rb * rows for (_, rb, rows, _) in self.regions)

    def dest_region(self, i: int) -> Region:
        """Where region i lands: the same rows and width at the destination offset and pitch."""
        off, rb, rows, pitch = self.regions[i]
        if self.dests is None:
            return self.regions[i]
        doff, dpitch = self.dests[i]
        return (doff, rb, rows, dpitch if rows > 1 else rb)

    def receivers(self, P: int, owner: int) -> List[int]:
        """The ranks this chunk is copied to (never its owner)."""
        return [q for q in range(P) if q != owner and (self.peers is None or (self.peers >> q) & 1)]


@dataclass
class Schedule:
    chunks: List[Chunk] = field(default_factory=list)

    @property
    def n_chunks(self) -> int:
        return len(self.chunks)

    @property
    def n_regions(self) -> int:
        return sum(len(c.regions) for c in self.chunks)


class ScheduleError(ValueError):
    """Invalid builder arguments."""


class PlanError(ValueError):
    """A plan the pages say must be rejected at creation; ``code`` names the reason."""

    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


def split_linear(offset: int, nbytes: int) -> List[Region]:
    """A byte range as linear copies of at most 1 GiB, full pieces first."""
    out = []
    pos = 0
    while pos < nbytes:
        n = min(LINEAR_MAX, nbytes - pos)
        out.append((offset + pos, n, 1, n))
        pos += n
    return out


def block_regions(offset: int, rows: int, row_bytes: int, pitch: int) -> List[Region]:
    """Regions for ``rows`` rows of ``row_bytes`` bytes, ``pitch`` bytes apart.

    Contiguous rows (pitch == row_bytes, or a single row) form one byte range split at 1 GiB;
    otherwise the rows form one 2D sub-window.
    """
    if rows == 0 or row_bytes == 0:
        return []
    if rows == 1 or pitch == row_bytes:
        return split_linear(offset, rows * row_bytes)
    return [(offset, row_bytes, rows, pitch)]


def whole(base_off: int, rows: int, row_bytes: int, pitch: int, num_programs: int) -> Schedule:
    if num_programs < 1:
        raise ScheduleError("num_programs must be >= 1")
    return Schedule([Chunk(block_regions(base_off, rows, row_bytes, pitch), num_programs)])


def chunks(base_off: int, rows: int, row_bytes: int, pitch: int, n: int) -> Schedule:
    if n < 1 or n > rows:
        raise ScheduleError("need 1 <= n <= rows")
    block = -(-rows // n)
    out = []
    r0 = 0
    while r0 < rows:
        nr = min(block, rows - r0)
        out.append(Chunk(block_regions(base_off + r0 * pitch, nr, row_bytes, pitch), 1))
        r0 += nr
    return Schedule(out)


def order_row_major(step: int, tiles_m: int, tiles_n: int) -> Tuple[int, int]:
    return step // tiles_n, step % tiles_n


def order_grouped(step: int, tiles_m: int, tiles_n: int, group_m: int) -> Tuple[int, int]:
    """Grouped step-to-tile order: GROUP_M tile rows are swept column by column.

    Reading of the elided ``tile_of(step, tiles_m, tiles_n, GROUP_M)``: steps fill groups of
    ``group_m`` consecutive tile rows; within a group, consecutive steps walk down the group's
    rows, then move one tile column right.  The last group may hold fewer rows.
    """
    per_group = group_m * tiles_n
    g = step // per_group
    m0 = g * group_m
    rows_in_group = min(tiles_m - m0, group_m)
    within = step % per_group
    return m0 + within % rows_in_group, within // rows_in_group


def tile_chunks(base_off: int, M: int, N: int, elem_bytes: int, pitch: int, BM: int, BN: int,
                tiles_per_chunk: int,
                order: Optional[Callable[[int], Tuple[int, int]]] = None) -> Schedule:
    if min(M, N, BM, BN, tiles_per_chunk, elem_bytes) < 1:
        raise ScheduleError("sizes must be positive")
    tiles_m = -(-M // BM)
    tiles_n = -(-N // BN)
    T = tiles_m * tiles_n
    if order is None:
        order = lambda s: order_row_major(s, tiles_m, tiles_n)  # noqa: E731
    seen = np.zeros((tiles_m, tiles_n), dtype=bool)
    regions = []
    for s in range(T):
        tm, tn = order(s)
        if not (0 <= tm < tiles_m and 0 <= tn < tiles_n) or seen[tm, tn]:
            raise ScheduleError("order is not a bijection onto the tiles")
        seen[tm, tn] = True
        rows = min(BM, M - tm * BM)
        cols = min(BN, N - tn * BN)
        regions.append((base_off + tm * BM * pitch + tn * BN * elem_bytes,
                        cols * elem_bytes, rows, pitch))
    out = []
    for k in range(0, T, tiles_per_chunk):
        steps = regions[k:k + tiles_per_chunk]
        out.append(Chunk(steps, len(steps)))
    return Schedule(out)


def first_chunks(schedules: Sequence[Schedule]) -> List[int]:
    """Global id of each rank's first chunk: the chunk counts of lower ranks, summed."""
    out, acc = [], 0
    for s in schedules:
        out.append(acc)
        acc += s.n_chunks
    return out


def region_extent(reg: Region) -> Tuple[int, int]:
    """Half-open byte span [lo, hi) touched by a region."""
    off, rb, rows, pitch = reg
    if rows == 0 or rb == 0:
        return off, off
    return off, off + (rows - 1) * pitch + rb


def region_byte_mask(reg: Region, nbytes: int) -> np.ndarray:
    """Boolean map of the bytes a region covers (brute force, for small buffers)."""
    m = np.zeros(nbytes, dtype=bool)
    off, rb, rows, pitch = reg
    for i in range(rows):
        m[off + i * pitch: off + i * pitch + rb] = True
    return m


def validate(schedules: Sequence[Schedule], buf_bytes: int, allgather: bool,
             max_regions: Optional[int] = None, dst_bytes: Optional[int] = None) -> None:
    """Reject a plan the pages say must not be created (raises PlanError).

    * every region lies inside the buffer;
    * all-gather: rank r's regions lie inside its own rows, bytes [r*S, (r+1)*S) with
      S = buf_bytes / P;
    * no byte is sent by two ranks to the same offsets (checked byte by byte);
    * optional capacity: at most ``max_regions`` regions in the plan;
    * destinations (see the module notes): inside the destination buffer (``dst_bytes`` when the
      plan has separate destination buffers, else the buffer), no two copies on the same bytes
      of one buffer, and in place no copy on bytes its receiving rank sends.
    """
    _validate_sources(schedules, buf_bytes, allgather, max_regions)
    _validate_destinations(schedules, buf_bytes, dst_bytes)


def _validate_destinations(schedules: Sequence[Schedule], buf_bytes: int,
                           dst_bytes: Optional[int]) -> None:
    P = len(schedules)
    nbytes = buf_bytes if dst_bytes is None else dst_bytes
    for r, sch in enumerate(schedules):
        for ch in sch.chunks:
            if ch.dests is not None and len(ch.dests) != len(ch.regions):
                raise PlanError("EINVAL", "one destination per region")
            if ch.peers is not None and (ch.peers >> P):
                raise PlanError("EINVAL", "peer mask names a rank outside the plan")
    for q in range(P):
        landed = np.zeros(nbytes, dtype=bool)
        if dst_bytes is None:            # in place: q's own sent bytes are not to be overwritten
            for ch in schedules[q].chunks:
                for reg in ch.regions:
                    landed |= region_byte_mask(reg, nbytes)
        for r, sch in enumerate(schedules):
            for ch in sch.chunks:
                if q not in ch.receivers(P, r):
                    continue
                for i in range(len(ch.regions)):
                    d = ch.dest_region(i)
                    doff, rb, rows, dpitch = d
                    if rows > 1 and dpitch < rb:
                        raise PlanError("EINVAL", "destination rows overlap (pitch < row_bytes)")
                    lo, hi = region_extent(d)
                    if lo < 0 or hi > nbytes:
                        raise PlanError("EINVAL", "destination outside the buffer")
                    m = region_byte_mask(d, nbytes)
                    if np.any(landed & m):
                        raise PlanError("EOVERLAP", f"two copies land on the same bytes of buffer {q}")
                    landed |= m


def _validate_sources(schedules: Sequence[Schedule], buf_bytes: int, allgather: bool,
                      max_regions: Optional[int]) -> None:
    P = len(schedules)
    if P < 1:
        raise PlanError("EINVAL", "no ranks")
    if allgather and buf_bytes % P:
        raise PlanError("EINVAL", "buffer does not split into P equal slices")
    S = buf_bytes // P if allgather else buf_bytes
    total = 0
    owner = np.full(buf_bytes, -1, dtype=np.int32)
    for r, sch in enumerate(schedules):
        for ch in sch.chunks:
            if ch.writers < 1:
                raise PlanError("EINVAL", "chunk with no writers")
            for reg in ch.regions:
                total += 1
                off, rb, rows, pitch = reg
                if rows > 1 and pitch < rb:
                    raise PlanError("EINVAL", "rows overlap (pitch < row_bytes)")
                lo, hi = region_extent(reg)
                if lo < 0 or hi > buf_bytes:
                    raise PlanError("EINVAL", "region outside the buffer")
                if allgather and not (r * S <= lo and hi <= (r + 1) * S):
                    raise PlanError("EOUTOFROWS", f"rank {r} region outside its own rows")
                if ch.dests is not None:
                    continue        # lands elsewhere: the destination checks govern it
                m = region_byte_mask(reg, buf_bytes)
                clash = owner[m]
                if np.any((clash >= 0) & (clash != r)):
                    raise PlanError("EOVERLAP", f"rank {r} sends bytes another rank sends")
                owner[m] = r
    if max_regions is not None and total > max_regions:
        raise PlanError("ECAPACITY", "too many regions")
