"""Oracle: the triggered plan's round and gate semantics, sequential definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Restated from the Iris "Triggered Plans" page (sections Model, The kernel author's contract,
Memory ordering, Gates and rounds, Requirements and limits) and "Triggered SDMA Plans" (ROCm/iris
pull 573, section Design notes):

* Every chunk has a gate row; this model keeps, per virtual rank and per global chunk id, the
  words ready, arrival, completion, error and the writer counter.  Rows of a rank's own chunks
  use ready / completion / error / counter; rows of other ranks' chunks use arrival.
* mark_ready: the writer counter goes up by one.  When it reaches round * writers the gate opens
  (ready := round).  A count above round * writers records the round in ``error``.
* The copy engine keeps one queue per (source, peer), holding the source's chunks in schedule
  order.  A queue waits until the low 32 bits of ready are >= round, copies the chunk's regions
  to the same offsets in the peer's buffer, then adds one to the peer's arrival word (and, in
  this model, one to the source's completion word).  A queue never passes a closed gate:
  later chunks wait behind it (head-of-line order).
* wait(): this rank's chunks were marked exactly ``writers`` times this round (more is an
  error, fewer a timeout naming the short chunks) and arrived at every peer; every other chunk
  arrived here.
* Rounds start at 1, go up by one per next_round and are never reset: at most 2**32 - 1.
* close() in the middle of a round sends each chunk as it stands: gates not yet open are
  opened and the queues drain.
* Groups ("Triggered Plans", Not supported yet: "Waiting on a group" -- the page only names the
  missing feature: no single counter covers several chunks or several source ranks).  Reading:
  a group is a set of global chunk ids, possibly of several source ranks; each virtual rank keeps
  one counter per group that goes up by one whenever one of the group's chunks becomes readable
  at that rank -- another rank's chunk when its arrival is signalled there, the rank's own chunk
  when its gate opens.  Every chunk becomes readable once per round at every rank, so after R
  rounds the counter holds R * |group|, and a wait on the group passes when the counter reaches
  round * |group|: exactly when every chunk of the group is readable there this round.
* Overlapping rounds ("Triggered Plans", Not supported yet: "Overlapping rounds" -- wait() must
  return before next_round() prepares the next round).  Reading, for a plan made with
  ``overlap=True``: next_round() may also be called while the round is RUNNING; that round then
  stays in flight (pending) and the next one is PREPARED, so at most two rounds are in flight.
  Each (source, peer) queue serves the pending round's chunks before the new round's, each in
  schedule order, so it still never passes a closed gate.  Round R+1's producer may write the
  bytes of its chunk only once every copy of that chunk made in round R has landed (its
  completion word holds R * receivers: ``writable``); whoever reads what round R delivered is
  done before round R+1's producers start (the model has no readers).  wait() reports the
  pending round first.  Its check is the sequential one, except that a count above
  R * writers may come from round R+1's marks: an extra mark shows in the error word (the mark
  that passes its round's count records it), and that word alone reports EXTRA.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import schedule as S

READY, ARRIVAL, COMPLETION, ERROR, COUNTER = range(5)
NFIELDS = 5
ROUND_LIMIT = (1 << 32) - 1

OK, EXTRA, TIMEOUT = "OK", "EXTRA", "TIMEOUT"


class StateError(RuntimeError):
    pass


class RoundLimitError(RuntimeError):
    pass


def copy_region(src: np.ndarray, dst: np.ndarray, reg: S.Region,
                dest: Optional[S.Region] = None) -> None:
    """Copy one region between two byte buffers: to the same offsets, or to ``dest`` (the same
    rows and width at another offset and pitch)."""
    off, rb, rows, pitch = reg
    doff, _, _, dpitch = reg if dest is None else dest
    if rows == 0 or rb == 0:
        return
    if rows == 1:
        dst[doff:doff + rb] = src[off:off + rb]
        return
    sv = np.lib.stride_tricks.as_strided(src[off:off + (rows - 1) * pitch + rb], shape=(rows, rb),
                                         strides=(pitch, 1))
    dv = np.lib.stride_tricks.as_strided(dst[doff:doff + (rows - 1) * dpitch + rb], shape=(rows, rb),
                                         strides=(dpitch, 1))
    dv[...] = sv


class Plan:
    """P virtual ranks, each with a byte buffer, one schedule each, and a gate table each."""

    def __init__(self, bufs: Sequence[np.ndarray], schedules: Sequence[S.Schedule],
                 allgather: bool = True, initial_round: int = 1, validate: bool = True,
                 copy_data: bool = True, dst_bufs: Optional[Sequence[np.ndarray]] = None,
                 overlap: bool = False):
        self.P = len(bufs)
        if len(schedules) != self.P:
            raise ValueError("one schedule per rank")
        nbytes = len(bufs[0])
        if any(len(b) != nbytes for b in bufs):
            raise ValueError("symmetric buffers must have one size")
        if not (1 <= initial_round <= ROUND_LIMIT):
            raise ValueError("initial round out of range")
        if dst_bufs is not None and (len(dst_bufs) != self.P or any(len(b) != len(dst_bufs[0]) for b in dst_bufs)):
            raise ValueError("one destination buffer per rank, all of one size")
        if validate:
            S.validate(schedules, nbytes, allgather,
                       dst_bytes=None if dst_bufs is None else len(dst_bufs[0]))
        self.bufs = list(bufs)
        self.dst = list(dst_bufs) if dst_bufs is not None else self.bufs   # where copies land
        self.copy_data = copy_data      # False: gate bookkeeping only (large workloads)
        self.schedules = list(schedules)
        self.first = S.first_chunks(schedules)
        self.owner: List[int] = []
        self.chunks: List[S.Chunk] = []
        for r, sch in enumerate(schedules):
            for ch in sch.chunks:
                self.owner.append(r)
                self.chunks.append(ch)
        self.G = len(self.chunks)
        self.round = initial_round
        self.gates = np.zeros((self.P, self.G, NFIELDS), dtype=np.uint64)
        prior = initial_round - 1      # gates as they stand after `prior` completed rounds
        for c, ch in enumerate(self.chunks):
            s = self.owner[c]
            self.gates[s, c, READY] = prior
            self.gates[s, c, COUNTER] = prior * ch.writers
            self.gates[s, c, COMPLETION] = prior * len(ch.receivers(self.P, s))
            for p in ch.receivers(self.P, s):
                self.gates[p, c, ARRIVAL] = prior
        self.delivered = set()          # (round, chunk, peer) delivered in a round still in flight
        self.delivery_log: List[Tuple[int, int, int]] = []   # (source, peer, chunk) in order
        self.delivery_rounds: List[int] = []                 # the round of each of them
        self.overlap = overlap
        self.pending: Optional[int] = None   # overlap: a round still in flight behind this one
        self.state = "PREPARED"
        self.groups: List[List[int]] = []
        self.groups_of: List[List[int]] = [[] for _ in range(self.G)]   # chunk -> its groups
        self.group_counters = np.zeros((self.P, 0), dtype=np.uint64)
        self.started = False

    # -- groups -------------------------------------------------------------------
    def define_groups(self, groups: Sequence[Sequence[int]]) -> None:
        """Declare the groups (lists of global chunk ids; a chunk may be in several groups).
        Allowed once, before the first round starts; counters begin as after the completed
        rounds before the current one."""
        if self.started or self.groups:
            raise StateError("groups are defined once, before the first start")
        for g in groups:
            if not len(g) or len(set(g)) != len(g) or any(not (0 <= c < self.G) for c in g):
                raise ValueError("a group is a non-empty set of chunk ids of the plan")
        self.groups = [list(g) for g in groups]
        self.groups_of = [[] for _ in range(self.G)]
        for i, g in enumerate(self.groups):
            for c in g:
                self.groups_of[c].append(i)
        prior = self.round - 1
        self.group_counters = np.zeros((self.P, len(self.groups)), dtype=np.uint64)
        for q in range(self.P):
            for i in range(len(self.groups)):
                self.group_counters[q, i] = prior * self.group_size(q, i)

    def reaches(self, rank: int, c: int) -> bool:
        """Does chunk c become readable at rank: it is rank's own, or rank receives it?"""
        return self.owner[c] == rank or rank in self.chunks[c].receivers(self.P, self.owner[c])

    def group_size(self, rank: int, g: int) -> int:
        """Members of group g that become readable at rank each round."""
        return sum(1 for c in self.groups[g] if self.reaches(rank, c))

    def chunk_readable(self, rank: int, c: int) -> bool:
        """Has chunk c become readable at rank this round (own chunk: gate open; another
        rank's chunk: its arrival signalled here)?"""
        if self.owner[c] == rank:
            return self.gate_open(c)
        return int(self.gates[rank, c, ARRIVAL]) >= self.round

    def group_ready(self, rank: int, g: int) -> bool:
        """The one test a group wait makes: the rank's counter of group g >= round * (members
        that reach the rank; all of them unless chunks go to only some peers)."""
        return int(self.group_counters[rank, g]) >= self.round * self.group_size(rank, g)

    def _count_group(self, rank: int, c: int) -> None:
        for g in self.groups_of[c]:
            self.group_counters[rank, g] += 1

    def signal_arrival(self, s: int, p: int, c: int) -> None:
        """The end of one copy of chunk c from s to p: arrival at p, completion at s, and p's
        counters of the chunk's groups."""
        self.gates[p, c, ARRIVAL] += 1
        self.gates[s, c, COMPLETION] += 1
        self._count_group(p, c)

    # -- round ------------------------------------------------------------------
    def start(self) -> int:
        if self.state != "PREPARED":
            raise StateError(f"start in state {self.state}")
        self.state = "RUNNING"
        self.started = True
        return self.round

    def chunks_of(self, r: int) -> range:
        return range(self.first[r], self.first[r] + self.schedules[r].n_chunks)

    def mark_ready(self, rank: int, c: int, rnd: Optional[int] = None) -> None:
        """One writer's mark on chunk c (global id) of its own rank, made in round ``rnd`` (the
        current round by default; with overlap, the pending round's producers may still be
        marking)."""
        if self.owner[c] != rank:
            raise ValueError("a rank marks only its own chunks")
        rnd = self.round if rnd is None else rnd
        if rnd not in self.rounds_in_flight():
            raise StateError(f"a mark of round {rnd}, which is not in flight")
        row = self.gates[rank, c]
        row[COUNTER] += 1
        target = rnd * self.chunks[c].writers
        if row[COUNTER] == target:
            row[READY] = rnd
            self._count_group(rank, c)     # readable at its own rank from now on
        elif row[COUNTER] > target:
            row[ERROR] = max(int(row[ERROR]), rnd)

    def rounds_in_flight(self) -> List[int]:
        """Rounds whose producers may mark and whose copies may move: the pending round (with
        overlap) and the current one once started."""
        live = [] if self.pending is None else [self.pending]
        if self.state in ("RUNNING", "CLOSING"):
            live.append(self.round)
        return live

    def writable(self, rank: int, c: int, rnd: Optional[int] = None) -> bool:
        """May round ``rnd``'s producer write rank's own chunk c: has every copy of it made in
        round rnd - 1 landed (completion >= (rnd - 1) * receivers)?  Always true without
        overlap, where round rnd starts after round rnd - 1's wait."""
        if self.owner[c] != rank:
            raise ValueError("writable is asked of a rank's own chunk")
        rnd = self.round if rnd is None else rnd
        return int(self.gates[rank, c, COMPLETION]) >= (rnd - 1) * len(self.chunks[c].receivers(self.P, rank))

    def write_chunk(self, rank: int, c: int, data: np.ndarray, rnd: Optional[int] = None) -> None:
        """Round rnd's producer writes chunk c of its rank: every region of it takes its bytes
        from ``data`` (a buffer-sized array of that round's contents).  Refused while the chunk
        is not writable."""
        if not self.writable(rank, c, rnd):
            raise StateError(f"chunk {c} written before round {rnd}'s previous copies of it landed")
        for reg in self.chunks[c].regions:
            copy_region(data, self.bufs[rank], reg)

    def reusable(self, rank: int, c: int) -> bool:
        """Source side: has every copy of rank's own chunk c landed at every peer this round?
        ("Triggered SDMA Plans", API: the device view's ``reusable``, which the page only names;
        read here as the test on the gate row's completion word from its Design notes.)  Each
        delivery adds one to the source's completion word, so the chunk is reusable once the
        word holds round * (P - 1)."""
        if self.owner[c] != rank:
            raise ValueError("reusable is asked of a rank's own chunk")
        return int(self.gates[rank, c, COMPLETION]) >= self.round * len(self.chunks[c].receivers(self.P, rank))

    def gate_open(self, c: int, rnd: Optional[int] = None) -> bool:
        s = self.owner[c]
        return (int(self.gates[s, c, READY]) & 0xFFFFFFFF) >= (self.round if rnd is None else rnd)

    def queue_next(self, s: int, p: int) -> Optional[Tuple[int, int]]:
        """The head of queue (s, p): (round, chunk) of its next copy, or None when it has
        nothing left in flight.  The pending round's chunks come before the current round's."""
        for rnd in self.rounds_in_flight():
            for c in self.chunks_of(s):
                if p in self.chunks[c].receivers(self.P, s) and (rnd, c, p) not in self.delivered:
                    return rnd, c
        return None

    def deliver_one(self, s: int, p: int) -> bool:
        """One step of queue (s, p): copy its head chunk if that chunk's gate is open for its
        round (else the queue waits: head of line).  Returns whether a copy was made."""
        head = self.queue_next(s, p)
        if head is None:
            return False
        rnd, c = head
        if not self.gate_open(c, rnd):
            return False
        ch = self.chunks[c]
        if self.copy_data:
            for i, reg in enumerate(ch.regions):
                copy_region(self.bufs[s], self.dst[p], reg, ch.dest_region(i))
        self.signal_arrival(s, p, c)
        self.delivered.add((rnd, c, p))
        self.delivery_log.append((s, p, c))
        self.delivery_rounds.append(rnd)
        return True

    def copier_progress(self) -> int:
        """Run every (source, peer) queue as far as its gates allow; returns deliveries made.
        Queue (s, p) holds s's chunks addressed to p, in schedule order (with overlap: the
        pending round's, then the current round's)."""
        n = 0
        for s in range(self.P):
            for p in range(self.P):
                if p == s:
                    continue
                while self.deliver_one(s, p):
                    n += 1
        return n

    def check(self, R: int, counter_extra: bool = True) -> Tuple[str, List[int], List[int]]:
        """Round R's completion check: (status, short chunk ids, extra chunk ids).  With
        counter_extra False (a round checked while the next one's marks may already count),
        only the error word reports an extra mark."""
        extra, short = [], []
        for c, ch in enumerate(self.chunks):
            s = self.owner[c]
            cnt = int(self.gates[s, c, COUNTER])
            if (counter_extra and cnt > R * ch.writers) or int(self.gates[s, c, ERROR]) != 0:
                extra.append(c)
            elif cnt < R * ch.writers:
                short.append(c)
            elif any(int(self.gates[p, c, ARRIVAL]) < R for p in ch.receivers(self.P, s)):
                short.append(c)
        return (EXTRA if extra else TIMEOUT if short else OK), short, extra

    def wait(self) -> Tuple[str, List[int], List[int]]:
        """Completion check of the oldest round in flight; returns (status, short chunk ids,
        extra chunk ids).  A pending round (overlap) is checked first and leaves the state as it
        is; otherwise the current round is checked and the plan becomes DONE."""
        if self.pending is not None:
            R = self.pending
            res = self.check(R, counter_extra=False)
            self.pending = None
            self.delivered = {d for d in self.delivered if d[0] != R}
            if res[0] != OK:
                self.state = "FAILED"
            return res
        if self.state != "RUNNING":
            raise StateError(f"wait in state {self.state}")
        res = self.check(self.round)
        self.state = "DONE" if res[0] == OK else "FAILED"
        return res

    def next_round(self) -> int:
        """Advance to the next round: from DONE, or (overlap) from RUNNING with no other round
        in flight, which leaves the running round pending."""
        if self.state == "RUNNING" and self.overlap and self.pending is None:
            if self.round >= ROUND_LIMIT:
                raise RoundLimitError("a plan is limited to 2**32 - 1 rounds")
            self.pending = self.round
            self.round += 1
            self.state = "PREPARED"
            return self.round
        if self.state != "DONE":
            raise StateError(f"next_round in state {self.state}")
        if self.round >= ROUND_LIMIT:
            raise RoundLimitError("a plan is limited to 2**32 - 1 rounds")
        self.round += 1
        self.delivered = set()
        self.state = "PREPARED"
        return self.round

    def close(self) -> None:
        """Close; mid-round, gates not yet open are opened and chunks sent as they stand (with
        overlap, for the pending round and the running one)."""
        live = self.rounds_in_flight()
        if live:
            top = live[-1]
            for c in range(self.G):
                if not self.gate_open(c, top):
                    self.gates[self.owner[c], c, READY] = top
            self.copier_progress()
        self.pending = None
        self.state = "CLOSED"


def expected_allgather(P: int, M: int, N: int, dtype: str, seed: int, rnd: int,
                       elem_bytes: int) -> np.ndarray:
    """Closed form: every virtual rank's buffer is the concatenation of all ranks' slices."""
    from . import hashfill
    return np.concatenate([hashfill.fill_slice_bytes(dtype, seed, r, rnd, M, N)
                           for r in range(P)])
