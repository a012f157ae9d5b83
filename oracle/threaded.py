"""Oracle: the triggered-plan protocol with CPU threads as ranks.  TEST INFRASTRUCTURE ONLY.

The same protocol as ``oracle.plan`` (the Iris "Triggered Plans" page, sections Model, The
kernel author's contract, Gates and rounds), but run concurrently: one thread per producer
program of each virtual rank and one copier thread per (source, peer) queue.  Gate words are
updated under a lock (standing in for atomics); every wait polls a bounded number of times.
It exercises what the sequential model cannot: head-of-line order on a queue when chunks
complete out of order (still correct, only slower), a missing mark (the queue times out and
wait() names the short chunk), an extra mark (wait() reports it) and close() in mid-round
(chunks are sent as they stand).  Nothing here touches a GPU.
"""
from __future__ import annotations

import threading
import time
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

from . import schedule as S
from .plan import READY, Plan, copy_region


class ThreadedRound:
    """Run one round of ``plan`` with threads.

    ``write_unit(rank, chunk, unit)`` stores writer ``unit`` of ``chunk`` into rank's buffer;
    ``order[rank]`` lists that rank's (chunk, unit) steps in the order its producer performs
    them (spread over ``programs`` threads round-robin); ``skip`` / ``extra`` name (chunk,
    unit) steps whose mark is dropped / doubled; ``delay`` gives per-step sleeps in seconds.
    """

    def __init__(self, plan: Plan, write_unit: Callable[[int, int, int], None],
                 order: Dict[int, List], programs: int = 1, max_polls: int = 20000,
                 poll_sleep: float = 1e-5, skip=(), extra=(), delay: Optional[Dict] = None,
                 group_waits: Sequence = ()):
        self.plan = plan
        self.write_unit = write_unit
        self.order = order
        self.programs = programs
        self.max_polls = max_polls
        self.poll_sleep = poll_sleep
        self.skip = set(skip)
        self.extra = set(extra)
        self.delay = delay or {}
        self.lock = threading.Lock()
        self.queue_log: Dict[tuple, List[int]] = {}
        self.timeouts: List[tuple] = []
        self.abort = threading.Event()
        # consumers: (rank, group) pairs, each a thread that waits once on the group and then
        # reads every chunk of it from the rank's own buffer; result per pair: "ok", "timeout"
        # or "stale" (a chunk's bytes differ from its source's)
        self.group_waits = list(group_waits)
        self.consumer_results: Dict[tuple, str] = {}

    # atomics --------------------------------------------------------------------------------
    def _mark(self, rank: int, c: int) -> None:
        with self.lock:
            self.plan.mark_ready(rank, c)

    def _ready(self, c: int) -> bool:
        with self.lock:
            return self.plan.gate_open(c)

    # threads ----------------------------------------------------------------------------------
    def _producer(self, rank: int, prog: int) -> None:
        for i, (c, u) in enumerate(self.order.get(rank, [])):
            if i % self.programs != prog:
                continue
            d = self.delay.get((c, u))
            if d:
                time.sleep(d)
            self.write_unit(rank, c, u)
            if (c, u) in self.skip:
                continue
            self._mark(rank, c)
            if (c, u) in self.extra:
                self._mark(rank, c)

    def _copier(self, s: int, p: int) -> None:
        plan = self.plan
        log = self.queue_log.setdefault((s, p), [])
        for c in plan.chunks_of(s):
            if p not in plan.chunks[c].receivers(plan.P, s):
                continue                    # not on this queue
            polls = 0
            while not self._ready(c):
                polls += 1
                if polls > self.max_polls or self.abort.is_set():
                    with self.lock:
                        self.timeouts.append((s, p, c))
                    return
                time.sleep(self.poll_sleep)
            ch = plan.chunks[c]
            for i, reg in enumerate(ch.regions):
                copy_region(plan.bufs[s], plan.dst[p], reg, ch.dest_region(i))
            with self.lock:
                plan.signal_arrival(s, p, c)
                plan.delivered.add((c, p))
            log.append(c)

    def _consumer(self, rank: int, g: int) -> None:
        plan = self.plan
        polls = 0
        while True:
            with self.lock:
                if plan.group_ready(rank, g):
                    break
            polls += 1
            if polls > self.max_polls or self.abort.is_set():
                self.consumer_results[(rank, g)] = "timeout"
                return
            time.sleep(self.poll_sleep)
        ok = True
        for c in plan.groups[g]:
            s = plan.owner[c]
            if s == rank or not plan.reaches(rank, c):
                continue                    # its own bytes, or not addressed to this rank
            ch = plan.chunks[c]
            for j, (off, nb, rows, pitch) in enumerate(ch.regions):
                doff, _, _, dpitch = ch.dest_region(j)
                for i in range(rows):
                    a, d = off + i * pitch, doff + i * dpitch
                    ok = ok and bool(np.array_equal(plan.dst[rank][d:d + nb], plan.bufs[s][a:a + nb]))
        self.consumer_results[(rank, g)] = "ok" if ok else "stale"

    def run(self, close_after: Optional[float] = None):
        """Start every thread, optionally close mid-round after ``close_after`` s, join, wait()."""
        plan = self.plan
        plan.start()
        threads = []
        for s in range(plan.P):
            for p in range(plan.P):
                if p != s:
                    threads.append(threading.Thread(target=self._copier, args=(s, p)))
        for (rank, g) in self.group_waits:
            threads.append(threading.Thread(target=self._consumer, args=(rank, g)))
        for r in range(plan.P):
            for q in range(self.programs):
                threads.append(threading.Thread(target=self._producer, args=(r, q)))
        for t in threads:
            t.start()
        if close_after is not None:
            time.sleep(close_after)
            with self.lock:                 # close(): open every gate as it stands
                for c in range(plan.G):
                    if not plan.gate_open(c):
                        plan.gates[plan.owner[c], c, READY] = plan.round
        for t in threads:
            t.join()
        if close_after is not None:
            plan.state = "CLOSED"
            return None
        return plan.wait()


def barrier_threads(P: int, gen_calls: int = 1, max_polls: int = 100000) -> np.ndarray:
    """The hand-rolled barrier with one thread per rank; returns each rank's final column."""
    signal = np.zeros((P, P), dtype=np.int64)
    lock = threading.Lock()
    ys = np.zeros((P, P), dtype=np.int64)
    failed = []

    def rank(r: int) -> None:
        for gen in range(1, gen_calls + 1):
            for peer in range(P):
                if peer != r:
                    with lock:
                        signal[peer, r] += 1          # AtomicAdd into row r of the peer
            for src in range(P):
                if src == r:
                    continue
                polls = 0
                while True:
                    with lock:
                        if signal[r, src] >= gen:     # Ge with a per-generation threshold
                            break
                    polls += 1
                    if polls > max_polls:
                        failed.append((r, src))
                        return
                    time.sleep(1e-6)
        with lock:
            ys[r] = signal[r]

    ts = [threading.Thread(target=rank, args=(r,)) for r in range(P)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if failed:
        raise RuntimeError(f"barrier waits timed out: {failed}")
    return ys
