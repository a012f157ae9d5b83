"""Pins for the oracle's overlapping rounds (oracle/plan.py, ``overlap=True``).

"Triggered Plans", Not supported yet: "Overlapping rounds" names the missing feature: wait()
must return before next_round() prepares the next round.  The oracle's reading lets round R+1
start while round R is in flight, as long as round R+1's producer writes a chunk only once
round R's copies of it have landed.  These tests pin that reading with facts that do not
depend on the model:
- the closed form of the all-gather after K rounds run two at a time;
- every copy carries the bytes of the round it is made in, over every interleaving of
  producers, queues and host calls on a small plan (exhaustive search);
- the same search finds torn copies once the writable rule is taken out of the oracle, so the
  search is able to see the mistake the rule prevents;
- hand-worked check results (an extra mark, a missing mark) while the next round's marks
  already count.
"""
import numpy as np
import pytest

from oracle import hashfill as H
from oracle import plan as PL
from oracle import schedule as S
from oracle.plan import ARRIVAL, COMPLETION, COUNTER, ERROR, READY


def _plan(P, M, N, n, writers=1, overlap=True, e=2):
    rb = N * e
    sb = M * rb
    bufs = [np.zeros(P * sb, dtype=np.uint8) for _ in range(P)]
    scheds = []
    for r in range(P):
        rows = -(-M // n)
        chunks = [S.Chunk([(r * sb + i * rows * rb, min(rows, M - i * rows) * rb, 1, min(rows, M - i * rows) * rb)],
                          writers) for i in range(n) if i * rows < M]
        scheds.append(S.Schedule(chunks))
    return PL.Plan(bufs, scheds, allgather=True, overlap=overlap), sb


def _round_data(P, sb, seed, R, M, N):
    """Each rank's buffer-sized array holding its round-R slice (hashed values) at its rows."""
    out = []
    for r in range(P):
        d = np.zeros(P * sb, dtype=np.uint8)
        d[r * sb:(r + 1) * sb] = H.fill_slice_bytes("bf16", seed, r, R, M, N)
        out.append(d)
    return out


@pytest.mark.parametrize("P,M,N,n,writers", [(2, 8, 16, 2, 1), (3, 12, 8, 4, 2), (4, 6, 4, 3, 1)])
def test_overlapped_rounds_closed_form(P, M, N, n, writers):
    # rounds started two at a time: round R's producers run while round R-1's copies are in
    # flight, each write waiting (here: the copier stepping) until the chunk is writable
    seed, K = 5, 5
    o, sb = _plan(P, M, N, n, writers)
    for R in range(1, K + 1):
        assert o.start() == R
        data = _round_data(P, sb, seed, R, M, N)
        for r in range(P):
            for c in o.chunks_of(r):
                steps = 0
                while not o.writable(r, c):
                    assert any(o.deliver_one(s, p) for s in range(P) for p in range(P) if p != s)
                    steps += 1
                assert steps == 0 or R > 1
                o.write_chunk(r, c, data[r])
                for _ in range(writers):
                    o.mark_ready(r, c)
        if o.pending is not None:
            o.copier_progress()
            assert o.wait() == (PL.OK, [], [])      # round R - 1
            assert o.state == "RUNNING" and o.round == R
        if R < K:
            assert o.next_round() == R + 1 and o.pending == R and o.state == "PREPARED"
    o.copier_progress()
    assert o.wait() == (PL.OK, [], []) and o.state == "DONE"
    want = np.concatenate([H.fill_slice_bytes("bf16", seed, r, K, M, N) for r in range(P)])
    for q in range(P):
        np.testing.assert_array_equal(o.bufs[q], want)
    for c in range(o.G):
        s = o.owner[c]
        assert o.gates[s, c, READY] == K and o.gates[s, c, COUNTER] == K * writers
        assert o.gates[s, c, COMPLETION] == K * (P - 1) and o.gates[s, c, ERROR] == 0
        assert all(o.gates[q, c, ARRIVAL] == K for q in range(P) if q != s)


# ---- exhaustive interleavings ----------------------------------------------------------------
# Two ranks, two chunks each, one writer, rounds 1 and 2 in flight together.  Processes:
#   producer r: round 1's chunks then round 2's, each a write and its mark; round 2's start only
#     after the host's next_round + start (and, being one stream, after round 1's);
#   queue (s, p): one copy per step, as the oracle's queue allows it;
#   host: next_round + start at any time; wait for round 1 once its copies have all landed.
# Each chunk holds 8 bytes = 4 bf16 of rank r's hashed values for its round.

def _explore(skip_writable):
    P, M, N = 2, 4, 1
    sb = M * 2
    seed = 3
    data = {R: _round_data(P, sb, seed, R, M, N) for R in (1, 2)}
    prod = [(R, c_local) for R in (1, 2) for c_local in range(2)]   # each producer's steps

    def fresh():
        o, _ = _plan(P, M, N, 2)
        o.start()
        return o

    violations, finals = [], 0
    seen = set()

    def key(o, pos, host):
        return (tuple(pos), host, o.round, o.pending, o.state,
                tuple(sorted(o.delivered)), b"".join(b.tobytes() for b in o.bufs), o.gates.tobytes())

    def clone(o):
        c = PL.Plan.__new__(PL.Plan)
        c.__dict__.update(o.__dict__)
        c.bufs = [b.copy() for b in o.bufs]
        c.dst = c.bufs
        c.gates = o.gates.copy()
        c.delivered = set(o.delivered)
        c.delivery_log = list(o.delivery_log)
        c.delivery_rounds = list(o.delivery_rounds)
        return c

    def moves(o, pos, host):
        out = []
        for r in range(P):
            if pos[r] < len(prod):
                R, cl = prod[pos[r]]
                c = o.first[r] + cl
                if R == 2 and host < 1:
                    continue                     # launched after the host starts round 2
                if not skip_writable and not o.writable(r, c, R):
                    continue                     # its wait for round R-1's copies of c
                out.append(("prod", r))
        for s in range(P):
            for p in range(P):
                if p != s:
                    head = o.queue_next(s, p)
                    if head is not None and o.gate_open(head[1], head[0]):
                        out.append(("copy", s, p))
        if host == 0:
            out.append(("next",))
        if host == 1 and o.pending == 1 and all((1, c, q) in o.delivered for c in range(o.G)
                                                for q in range(P) if q != o.owner[c]):
            out.append(("wait1",))
        return out

    def apply(o, pos, host, m):
        o = clone(o)
        pos = list(pos)
        if m[0] == "prod":
            r = m[1]
            R, cl = prod[pos[r]]
            c = o.first[r] + cl
            for reg in o.chunks[c].regions:          # the write, with or without the rule
                PL.copy_region(data[R][r], o.bufs[r], reg)
            o.mark_ready(r, c, R)
            pos[r] += 1
        elif m[0] == "copy":
            _, s, p = m
            R, c = o.queue_next(s, p)
            assert o.deliver_one(s, p)
            off, n, _, _ = o.chunks[c].regions[0]
            if not np.array_equal(o.bufs[p][off:off + n], data[R][s][off:off + n]):
                violations.append((R, s, p, c))
        elif m[0] == "next":
            assert o.next_round() == 2
            o.start()
            host = 1
        else:
            assert o.wait() == (PL.OK, [], [])
            host = 2
        return o, pos, host

    stack = [(fresh(), [0, 0], 0)]
    while stack:
        o, pos, host = stack.pop()
        k = key(o, pos, host)
        if k in seen:
            continue
        seen.add(k)
        ms = moves(o, pos, host)
        if not ms:
            # everything produced and copied: round 2's wait and its closed form
            assert pos == [len(prod)] * P and host == 2, (pos, host)
            o.copier_progress()
            assert o.wait()[0] == PL.OK
            want = np.concatenate([H.fill_slice_bytes("bf16", seed, r, 2, M, N) for r in range(P)])
            finals += 1
            if not all(np.array_equal(b, want) for b in o.bufs):
                violations.append(("final",))
            continue
        for m in ms:
            stack.append(apply(o, pos, host, m))
    return violations, finals, len(seen)


def test_every_interleaving_copies_each_rounds_own_bytes():
    violations, finals, states = _explore(skip_writable=False)
    assert violations == []
    assert finals >= 1 and states > 100


def test_search_finds_torn_copies_without_the_writable_rule():
    # the mistake planted in the oracle: round 2's producer writes a chunk without waiting for
    # round 1's copy of it; some interleaving then copies round 2's bytes in round 1
    violations, _, _ = _explore(skip_writable=True)
    assert any(v[0] == 1 for v in violations)


# ---- the check while the next round counts ------------------------------------------------------

def test_extra_mark_is_reported_by_its_rounds_wait():
    # round 1: chunk 0 of rank 0 gets 2 marks for 1 writer (counter 2 > 1, error = 1).  Round 2
    # then runs on the other chunks; round 1's wait reports chunk 0 as EXTRA
    o, sb = _plan(2, 4, 4, 2)
    o.start()
    for r in range(2):
        for c in o.chunks_of(r):
            o.mark_ready(r, c)
    o.mark_ready(0, 0)
    assert o.gates[0, 0, COUNTER] == 2 and o.gates[0, 0, ERROR] == 1
    o.next_round()
    o.start()
    o.copier_progress()
    assert o.wait() == (PL.EXTRA, [], [0]) and o.state == "FAILED"


def test_next_rounds_marks_are_not_extra_marks():
    # round 2 marks chunk 1 of rank 0 (writable once round 1's copy of it landed) before round
    # 1's wait: the counter reads 2 > 1 * writers, and round 1 is still OK
    o, sb = _plan(2, 4, 4, 2)
    o.start()
    for r in range(2):
        for c in o.chunks_of(r):
            o.mark_ready(r, c)
    o.next_round()
    o.start()
    o.copier_progress()
    assert o.writable(0, 1)
    o.mark_ready(0, 1)
    assert o.gates[0, 1, COUNTER] == 2 and o.gates[0, 1, READY] == 2
    assert o.wait() == (PL.OK, [], [])
    assert o.state == "RUNNING" and o.pending is None


def test_missing_mark_is_short_and_its_chunk_never_writable():
    o, sb = _plan(2, 4, 4, 2)
    o.start()
    for r in range(2):
        for c in o.chunks_of(r):
            if c != 1:
                o.mark_ready(r, c)
    o.next_round()
    o.start()
    o.copier_progress()
    assert not o.writable(0, 1) and o.writable(0, 0)
    with pytest.raises(PL.StateError):
        o.write_chunk(0, 1, np.zeros(len(o.bufs[0]), dtype=np.uint8))
    assert o.wait() == (PL.TIMEOUT, [1], []) and o.state == "FAILED"


def test_overlap_state_rules():
    o, sb = _plan(2, 4, 4, 2)
    o.start()
    o.next_round()
    with pytest.raises(PL.StateError):
        o.next_round()                    # PREPARED, and round 1 still in flight
    o.start()
    with pytest.raises(PL.StateError):
        o.next_round()                    # two rounds in flight already
    with pytest.raises(PL.StateError):
        o.mark_ready(0, 0, 3)             # round 3 is not in flight
    seq, _ = _plan(2, 4, 4, 2, overlap=False)
    seq.start()
    with pytest.raises(PL.StateError):
        seq.next_round()                  # without overlap: only from DONE
    # close with two rounds in flight opens both rounds' gates and drains every queue
    o.close()
    assert o.state == "CLOSED"
    assert all(o.gates[o.owner[c], c, READY] == 2 for c in range(o.G))
    assert all(o.gates[q, c, ARRIVAL] == 2 for c in range(o.G) for q in range(2) if q != o.owner[c])
