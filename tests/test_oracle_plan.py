"""Pins for the oracle's round and gate semantics (oracle/plan.py)."""
import itertools

import numpy as np
import pytest

from oracle import hashfill as H
from oracle import plan as PL
from oracle import schedule as S
from oracle.plan import ARRIVAL, COMPLETION, COUNTER, ERROR, READY


def make_plan(P, M, N, dtype, kind, initial_round=1, **kw):
    e = {"bf16": 2, "f32": 4, "u8": 1}[dtype]
    rb = N * e
    slice_bytes = M * rb
    bufs = [np.zeros(P * slice_bytes, dtype=np.uint8) for _ in range(P)]
    scheds = []
    for r in range(P):
        off = r * slice_bytes
        if kind == "whole":
            scheds.append(S.whole(off, M, rb, rb, kw.get("np", 1)))
        elif kind == "chunks":
            scheds.append(S.chunks(off, M, rb, rb, kw["n"]))
        else:
            tm, tn = -(-M // kw["BM"]), -(-N // kw["BN"])
            gm = kw.get("gm", 0)
            order = (lambda s, tm=tm, tn=tn: S.order_grouped(s, tm, tn, gm)) if gm else None
            scheds.append(S.tile_chunks(off, M, N, e, rb, kw["BM"], kw["BN"], kw["T"], order))
    return PL.Plan(bufs, scheds, allgather=True, initial_round=initial_round), slice_bytes


def produce_all(plan, P, M, N, dtype, seed, slice_bytes):
    """Each rank writes its slice for this round, then marks every chunk writers times."""
    for r in range(P):
        plan.bufs[r][r * slice_bytes:(r + 1) * slice_bytes] = \
            H.fill_slice_bytes(dtype, seed, r, plan.round, M, N)
        for c in plan.chunks_of(r):
            for _ in range(plan.chunks[c].writers):
                plan.mark_ready(r, c)


CASES = [
    (2, 8, 16, "bf16", "whole", {"np": 1}),
    (4, 12, 10, "f32", "chunks", {"n": 4}),
    (3, 10, 9, "bf16", "tile_chunks", {"BM": 4, "BN": 4, "T": 2, "gm": 2}),
    (2, 5, 7, "u8", "tile_chunks", {"BM": 2, "BN": 3, "T": 5}),
    (8, 4, 8, "f32", "whole", {"np": 8}),
]


@pytest.mark.parametrize("P,M,N,dtype,kind,kw", CASES)
def test_allgather_closed_form_and_gate_invariants(P, M, N, dtype, kind, kw):
    seed = 99
    plan, sb = make_plan(P, M, N, dtype, kind, **kw)
    e = {"bf16": 2, "f32": 4, "u8": 1}[dtype]
    for R in range(1, 4):
        assert plan.start() == R
        produce_all(plan, P, M, N, dtype, seed, sb)
        plan.copier_progress()
        assert plan.wait() == (PL.OK, [], [])
        want = PL.expected_allgather(P, M, N, dtype, seed, R, e)
        for q in range(P):
            assert np.array_equal(plan.bufs[q], want), (R, q)
        for c, ch in enumerate(plan.chunks):
            s = plan.owner[c]
            assert plan.gates[s, c, COUNTER] == R * ch.writers
            assert plan.gates[s, c, READY] == R
            assert plan.gates[s, c, COMPLETION] == R * (P - 1)
            assert plan.gates[s, c, ERROR] == 0
            for p in range(P):
                assert plan.gates[p, c, ARRIVAL] == (R if p != s else 0)
        # per source, arrivals summed over its chunks = round x chunks at every peer
        for s in range(P):
            for p in range(P):
                if p != s:
                    assert sum(int(plan.gates[p, c, ARRIVAL]) for c in plan.chunks_of(s)) == \
                        R * plan.schedules[s].n_chunks
        plan.next_round()


def test_extra_mark_is_reported_and_missing_mark_times_out():
    plan, sb = make_plan(2, 4, 4, "bf16", "chunks", n=2)
    plan.start()
    produce_all(plan, 2, 4, 4, "bf16", 1, sb)
    plan.mark_ready(1, 3)                   # one mark too many on rank 1's second chunk
    plan.copier_progress()
    status, short, extra = plan.wait()
    assert status == PL.EXTRA and extra == [3] and plan.gates[1, 3, ERROR] == 1
    assert plan.state == "FAILED"

    plan, sb = make_plan(2, 4, 4, "bf16", "chunks", n=2)
    plan.start()
    for r in range(2):
        for c in plan.chunks_of(r):
            if c != 1:
                plan.mark_ready(r, c)
    plan.copier_progress()
    status, short, extra = plan.wait()
    assert status == PL.TIMEOUT and short == [1] and extra == []
    assert plan.gates[0, 1, READY] == 0 and plan.gates[1, 1, ARRIVAL] == 0


def test_head_of_line_order():
    plan, sb = make_plan(2, 6, 4, "bf16", "chunks", n=3)
    plan.start()
    plan.mark_ready(0, 2)                   # rank 0 completes its last chunk first
    plan.mark_ready(0, 1)
    plan.copier_progress()
    assert plan.gates[1, 1, ARRIVAL] == 0 and plan.gates[1, 2, ARRIVAL] == 0
    plan.mark_ready(0, 0)
    plan.copier_progress()
    assert [c for (s, p, c) in plan.delivery_log if s == 0] == [0, 1, 2]


def test_round_limit():
    top = (1 << 32) - 1
    plan, sb = make_plan(2, 4, 4, "bf16", "whole", initial_round=top - 1)
    for R in (top - 1, top):
        assert plan.start() == R
        produce_all(plan, 2, 4, 4, "bf16", 5, sb)
        plan.copier_progress()
        assert plan.wait()[0] == PL.OK
        assert plan.gates[0, 0, READY] == R
        if R < top:
            plan.next_round()
    with pytest.raises(PL.RoundLimitError):
        plan.next_round()


def test_state_machine():
    plan, sb = make_plan(2, 4, 4, "bf16", "whole")
    with pytest.raises(PL.StateError):
        plan.wait()
    with pytest.raises(PL.StateError):
        plan.next_round()
    plan.start()
    with pytest.raises(PL.StateError):
        plan.start()


def test_close_mid_round_sends_chunks_as_they_stand():
    P, M, N = 2, 4, 8
    plan, sb = make_plan(P, M, N, "bf16", "chunks", n=2)
    plan.start()
    full = H.fill_slice_bytes("bf16", 4, 0, 1, M, N)
    plan.bufs[0][:sb // 2] = full[:sb // 2]            # rank 0 wrote only its first block
    plan.mark_ready(0, 0)
    plan.close()
    assert np.array_equal(plan.bufs[1][:sb], plan.bufs[0][:sb])
    assert np.all(plan.bufs[1][sb // 2:sb] == 0)        # second block went as it stood
    assert plan.state == "CLOSED"


def test_bytes_outside_regions_untouched():
    P, M, rb = 2, 4, 8
    bufs = [np.full(P * M * rb, 0xEE, dtype=np.uint8) for _ in range(P)]
    # each rank sends only the first 4 bytes of each of its rows (a 2D window)
    scheds = [S.Schedule([S.Chunk([(r * M * rb, 4, M, rb)], 1)]) for r in range(P)]
    plan = PL.Plan(bufs, scheds)
    plan.start()
    bufs[0][:M * rb] = 1
    bufs[1][M * rb:] = 2
    plan.mark_ready(0, 0)
    plan.mark_ready(1, 1)
    plan.copier_progress()
    assert plan.wait()[0] == PL.OK
    row = np.array([1] * 4 + [0xEE] * 4, dtype=np.uint8)
    assert np.array_equal(bufs[1][:M * rb], np.tile(row, M))
    row = np.array([2] * 4 + [0xEE] * 4, dtype=np.uint8)
    assert np.array_equal(bufs[0][M * rb:], np.tile(row, M))


def test_exhaustive_interleavings_tiny_plan():
    """P=2, two chunks per rank, two writers per chunk: every interleaving of the eight marks
    (each writer marks its two chunks in order, after writing its half of the chunk) with the
    copier running after every event.  The gate never opens before both writers' marks of the
    round, arrival never precedes ready, and every round ends with the closed-form buffers."""
    P, rb = 2, 8
    nrows = 4                                # per rank: 2 chunks x 2 rows
    sb = nrows * rb
    seqs = [(r, w) for r in range(P) for w in range(2)]     # four writers
    events = [x for x in seqs for _ in range(2)]
    orders = set(itertools.permutations(events))
    assert len(orders) == 2520
    for order in sorted(orders):
        bufs = [np.zeros(P * sb, dtype=np.uint8) for _ in range(P)]
        scheds = [S.Schedule([S.Chunk([(r * sb + k * 2 * rb, 2 * rb, 1, 2 * rb)], 2)
                              for k in range(2)]) for r in range(P)]
        plan = PL.Plan(bufs, scheds)
        for R in (1, 2):
            plan.start()
            pos = {x: 0 for x in seqs}
            for ev in order:
                r, w = ev
                k = pos[ev]
                pos[ev] += 1
                c = plan.first[r] + k
                lo = r * sb + k * 2 * rb + w * rb          # writer w's row of chunk k
                bufs[r][lo:lo + rb] = 16 * R + 4 * r + w
                plan.mark_ready(r, c)
                for cc in range(plan.G):
                    s = plan.owner[cc]
                    opened = int(plan.gates[s, cc, READY]) >= R
                    assert opened == (int(plan.gates[s, cc, COUNTER]) >= R * 2)
                plan.copier_progress()
                for cc in range(plan.G):
                    s = plan.owner[cc]
                    for p in range(P):
                        if p != s and int(plan.gates[p, cc, ARRIVAL]) >= R:
                            assert int(plan.gates[s, cc, READY]) >= R
            assert plan.wait()[0] == PL.OK
            for q in range(P):
                for r in range(P):
                    for k in range(2):
                        for w in range(2):
                            lo = r * sb + k * 2 * rb + w * rb
                            assert np.all(bufs[q][lo:lo + rb] == 16 * R + 4 * r + w)
            plan.next_round()


def test_reusable_is_delivered_to_every_peer_this_round():
    # reusable(c) holds exactly when chunk c has arrived at every other rank in this round: a
    # test of completion against P - 1 without the round, or against one peer's arrival, fails
    # in round 2 or before the last queue has delivered
    rng = np.random.default_rng(3)
    P = 3
    plan, sb = make_plan(P, 6, 4, "bf16", "chunks", n=3)
    for R in (1, 2, 3):
        plan.start()
        own = [(r, c) for r in range(P) for c in plan.chunks_of(r)]
        for r, c in own:
            assert not plan.reusable(r, c)          # nothing delivered yet this round
        marks = [(r, c) for r, c in own for _ in range(plan.chunks[c].writers)]
        for i in rng.permutation(len(marks)):
            r, c = marks[i]
            plan.mark_ready(r, c)
            if rng.random() < 0.5:
                plan.copier_progress()
            for r2, c2 in own:
                delivered = all(int(plan.gates[p, c2, ARRIVAL]) >= R for p in range(P) if p != r2)
                assert plan.reusable(r2, c2) == delivered
        plan.copier_progress()
        assert all(plan.reusable(r, c) for r, c in own)
        assert plan.wait()[0] == PL.OK
        plan.next_round()
    with pytest.raises(ValueError):
        plan.reusable(0, plan.first[1])               # a chunk of another rank


def test_reusable_follows_head_of_line_order():
    plan, sb = make_plan(2, 6, 4, "bf16", "chunks", n=3)
    plan.start()
    plan.mark_ready(0, 1)                  # chunk 1 is ready but queued behind chunk 0
    plan.copier_progress()
    assert not plan.reusable(0, 1) and not plan.reusable(0, 0)
    plan.mark_ready(0, 0)
    plan.copier_progress()
    assert plan.reusable(0, 0) and plan.reusable(0, 1) and not plan.reusable(0, 2)


# ---- groups ("Triggered Plans", Not supported yet: "Waiting on a group") ------------------------
def _random_groups(plan, rng, n):
    """n groups of random chunk sets, across source ranks; chunks may repeat across groups."""
    out = []
    for _ in range(n):
        k = int(rng.integers(1, plan.G + 1))
        out.append(sorted(int(c) for c in rng.choice(plan.G, size=k, replace=False)))
    return out


def test_group_counters_closed_form_after_each_round():
    # each chunk becomes readable once per round at every rank (its own rank: when its gate
    # opens), so after R rounds every rank's counter of group g holds R * |g|
    rng = np.random.default_rng(5)
    for P, kind, kw in [(3, "chunks", {"n": 3}), (4, "tile_chunks", {"BM": 2, "BN": 4, "T": 3}),
                        (2, "whole", {"np": 2})]:
        plan, sb = make_plan(P, 6, 8, "bf16", kind, **kw)
        groups = _random_groups(plan, rng, 5) + [list(range(plan.G))]
        plan.define_groups(groups)
        for R in (1, 2, 3):
            plan.start()
            produce_all(plan, P, 6, 8, "bf16", 1, sb)
            plan.copier_progress()
            assert plan.wait()[0] == PL.OK
            for q in range(P):
                for g, members in enumerate(groups):
                    assert int(plan.group_counters[q, g]) == R * len(members)
            plan.next_round()


def test_group_wait_passes_exactly_when_every_member_is_readable():
    # the definition of waiting on a group: every chunk of it readable at the rank this round.
    # Checked at every step of random mark orders with the copier run at random moments, in
    # rounds 1-3 (a test against |g| without the round, or of arrival only, fails here)
    rng = np.random.default_rng(9)
    P = 3
    plan, sb = make_plan(P, 6, 4, "bf16", "chunks", n=3)
    groups = _random_groups(plan, rng, 8) + [[plan.first[1]], [plan.first[0], plan.first[2] + 1]]
    plan.define_groups(groups)
    for R in (1, 2, 3):
        plan.start()
        marks = [(r, c) for r in range(P) for c in plan.chunks_of(r) for _ in range(plan.chunks[c].writers)]

        def check():
            for q in range(P):
                for g, members in enumerate(groups):
                    assert plan.group_ready(q, g) == all(plan.chunk_readable(q, c) for c in members)
        check()
        for i in rng.permutation(len(marks)):
            plan.mark_ready(*marks[i])
            check()
            if rng.random() < 0.4:
                plan.copier_progress()
                check()
        plan.copier_progress()
        check()
        assert all(plan.group_ready(q, g) for q in range(P) for g in range(len(groups)))
        assert plan.wait()[0] == PL.OK
        plan.next_round()


def test_group_of_own_chunks_opens_with_the_gates():
    # a rank's own chunks count when their gates open, not when they reach peers
    plan, sb = make_plan(2, 6, 4, "bf16", "chunks", n=3)
    plan.define_groups([list(plan.chunks_of(0)), [plan.first[0], plan.first[1]]])
    plan.start()
    for c in plan.chunks_of(0):
        plan.mark_ready(0, c)
    assert plan.group_ready(0, 0)                   # no copy needed for rank 0's own chunks
    assert not plan.group_ready(1, 0)               # nothing copied yet
    plan.copier_progress()
    assert plan.group_ready(1, 0)
    assert not plan.group_ready(0, 1) and not plan.group_ready(1, 1)   # rank 1's chunk 0 not marked
    plan.mark_ready(1, plan.first[1])
    assert plan.group_ready(1, 1) and not plan.group_ready(0, 1)
    plan.copier_progress()
    assert plan.group_ready(0, 1)


def test_group_head_of_line_and_initial_round():
    # a group whose member waits behind a closed gate on its queue is not ready; counters of a
    # plan that begins at round R0 start as after R0 - 1 rounds
    plan, sb = make_plan(2, 6, 4, "bf16", "chunks", initial_round=7, n=3)
    plan.define_groups([[plan.first[0] + 1], [plan.first[0], plan.first[0] + 2]])
    assert list(plan.group_counters[:, 0]) == [6, 6] and list(plan.group_counters[:, 1]) == [12, 12]
    plan.start()
    plan.mark_ready(0, plan.first[0] + 1)           # queued behind chunk 0 on the way to rank 1
    plan.copier_progress()
    assert plan.group_ready(0, 0) and not plan.group_ready(1, 0)
    plan.mark_ready(0, plan.first[0])
    plan.copier_progress()
    assert plan.group_ready(1, 0) and not plan.group_ready(1, 1)


def test_group_definition_rules():
    plan, sb = make_plan(2, 6, 4, "bf16", "chunks", n=3)
    for bad in ([[]], [[0, 0]], [[plan.G]], [[-1]]):
        with pytest.raises(ValueError):
            plan.define_groups(bad)
    plan.define_groups([[0, 1]])
    with pytest.raises(PL.StateError):
        plan.define_groups([[0]])                   # once per plan
    plan2, _ = make_plan(2, 6, 4, "bf16", "chunks", n=3)
    plan2.start()
    with pytest.raises(PL.StateError):
        plan2.define_groups([[0]])                  # before the first start


def test_group_exhaustive_interleavings_tiny_plan():
    # P = 2, two chunks per rank with two writers each, one group of all four chunks and one of
    # the two ranks' first chunks: in every interleaving of the eight marks, with the copier run
    # after each, a group is ready at a rank exactly when each of its chunks is readable there
    P, rb = 2, 8
    sb = 4 * rb
    seqs = [(r, w) for r in range(P) for w in range(2)]
    events = [x for x in seqs for _ in range(2)]
    for order in sorted(set(itertools.permutations(events))):
        bufs = [np.zeros(P * sb, dtype=np.uint8) for _ in range(P)]
        scheds = [S.Schedule([S.Chunk([(r * sb + k * 2 * rb, 2 * rb, 1, 2 * rb)], 2)
                              for k in range(2)]) for r in range(P)]
        plan = PL.Plan(bufs, scheds)
        groups = [[0, 1, 2, 3], [0, 2]]
        plan.define_groups(groups)
        plan.start()
        pos = {x: 0 for x in seqs}
        for ev in order:
            r, w = ev
            k = pos[ev]
            pos[ev] += 1
            plan.mark_ready(r, plan.first[r] + k)
            plan.copier_progress()
            for q in range(P):
                for g, members in enumerate(groups):
                    assert plan.group_ready(q, g) == all(plan.chunk_readable(q, c) for c in members)
        assert all(plan.group_ready(q, g) for q in range(P) for g in range(2))


# ---- other destinations ("Triggered Plans", Not supported yet: "Other destinations") ---------------
def _reduce_scatter_plan(P, B, dst_bufs=False, initial_round=1):
    """Rank s holds P partial blocks of B bytes at [0, P*B) and a staging area of P slots at
    [P*B, 2*P*B).  Chunk b of rank s is its partial block b, sent only to rank b, landing in
    rank b's staging slot s (or in rank b's separate destination buffer, slot s)."""
    nbytes = 2 * P * B
    bufs = [np.zeros(nbytes, dtype=np.uint8) for _ in range(P)]
    dst = [np.zeros(P * B, dtype=np.uint8) for _ in range(P)] if dst_bufs else None
    scheds = []
    for s in range(P):
        chunks = []
        for b in range(P):
            if b == s:
                continue
            slot = (s * B) if dst_bufs else (P * B + s * B)
            chunks.append(S.Chunk([(b * B, B, 1, B)], 1, dests=[(slot, B)], peers=1 << b))
        scheds.append(S.Schedule(chunks))
    plan = PL.Plan(bufs, scheds, allgather=False, initial_round=initial_round, dst_bufs=dst)
    return plan


@pytest.mark.parametrize("dst_bufs", [False, True])
def test_reduce_scatter_staging_closed_form(dst_bufs):
    # every rank's partial for block b lands in rank b's slot of its own rank number, nowhere
    # else; arrivals only at the receiver; completion counts one receiver per chunk
    P, B = 4, 16
    plan = _reduce_scatter_plan(P, B, dst_bufs)
    for R in (1, 2, 3):
        plan.start()
        for s in range(P):
            plan.bufs[s][:P * B] = (np.arange(P * B) * 7 + 31 * s + 101 * R) % 251
            for c in plan.chunks_of(s):
                plan.mark_ready(s, c)
        plan.copier_progress()
        assert plan.wait()[0] == PL.OK
        for b in range(P):
            base = 0 if dst_bufs else P * B
            out = plan.dst[b]
            for s in range(P):
                slot = out[base + s * B: base + (s + 1) * B]
                if s == b:
                    assert np.all(slot == 0)                  # nothing lands in one's own slot
                else:
                    assert np.array_equal(slot, plan.bufs[s][b * B:(b + 1) * B])
        for c in range(plan.G):
            s = plan.owner[c]
            (b,) = plan.chunks[c].receivers(P, s)
            for q in range(P):
                assert int(plan.gates[q, c, ARRIVAL]) == (R if q == b else 0)
            assert int(plan.gates[s, c, COMPLETION]) == R
        plan.next_round()


def test_pitched_destination_lands_row_by_row():
    # a 2D window of 3 rows x 8 bytes (source pitch 16) lands with destination pitch 40
    src_reg, dest = (4, 8, 3, 16), (100, 40)
    bufs = [np.zeros(256, dtype=np.uint8) for _ in range(2)]
    scheds = [S.Schedule([S.Chunk([src_reg], 1, dests=[dest])]), S.Schedule()]
    plan = PL.Plan(bufs, scheds, allgather=False)
    plan.start()
    bufs[0][:64] = np.arange(64)
    plan.mark_ready(0, 0)
    plan.copier_progress()
    assert plan.wait()[0] == PL.OK
    want = np.zeros(256, dtype=np.uint8)
    for i in range(3):
        want[100 + 40 * i:108 + 40 * i] = np.arange(4 + 16 * i, 12 + 16 * i)
    assert np.array_equal(bufs[1], want)


def test_queues_hold_only_their_peers_chunks():
    # rank 0's chunk 0 goes to rank 1 only and is never marked; chunk 1 goes to rank 2 only: it
    # is not behind chunk 0 on any queue, so it arrives; chunk 2 (to everyone) waits behind
    # chunk 0 on queue (0, 1) only
    B = 8
    bufs = [np.zeros(3 * 3 * B, dtype=np.uint8) for _ in range(3)]
    scheds = [S.Schedule([S.Chunk([(0, B, 1, B)], 1, peers=0b010), S.Chunk([(B, B, 1, B)], 1, peers=0b100),
                          S.Chunk([(2 * B, B, 1, B)], 1)]), S.Schedule(), S.Schedule()]
    plan = PL.Plan(bufs, scheds, allgather=False)
    plan.start()
    plan.mark_ready(0, 1)
    plan.mark_ready(0, 2)
    plan.copier_progress()
    assert int(plan.gates[2, 1, ARRIVAL]) == 1 and int(plan.gates[2, 2, ARRIVAL]) == 1
    assert int(plan.gates[1, 2, ARRIVAL]) == 0          # head of line behind chunk 0 on (0, 1)
    assert plan.reusable(0, 1) and not plan.reusable(0, 2)
    status, short, extra = plan.wait()
    assert status == PL.TIMEOUT and short == [0, 2]


def test_destination_validation():
    B = 8
    def plan_of(scheds, nbytes=64, dst=None):
        return PL.Plan([np.zeros(nbytes, dtype=np.uint8) for _ in range(len(scheds))], scheds,
                       allgather=False, dst_bufs=dst)
    # two ranks' copies land on the same bytes of rank 2
    with pytest.raises(S.PlanError) as e:
        plan_of([S.Schedule([S.Chunk([(0, B, 1, B)], 1, dests=[(40, B)], peers=0b100)]),
                 S.Schedule([S.Chunk([(B, B, 1, B)], 1, dests=[(44, B)], peers=0b100)]), S.Schedule()])
    assert e.value.code == "EOVERLAP"
    # in place, a copy onto bytes the receiving rank itself sends
    with pytest.raises(S.PlanError) as e:
        plan_of([S.Schedule([S.Chunk([(0, B, 1, B)], 1, dests=[(16, B)])]),
                 S.Schedule([S.Chunk([(16, B, 1, B)], 1, peers=0b01)])])
    assert e.value.code == "EOVERLAP"
    # ... allowed into separate destination buffers
    plan_of([S.Schedule([S.Chunk([(0, B, 1, B)], 1, dests=[(16, B)])]),
             S.Schedule([S.Chunk([(16, B, 1, B)], 1, peers=0b01)])], dst=[np.zeros(32, np.uint8)] * 2)
    for bad in (S.Chunk([(0, B, 1, B)], 1, dests=[(60, B)]),              # past the end
                S.Chunk([(0, B, 2, B)], 1, dests=[(0, B - 1)]),          # destination rows overlap
                S.Chunk([(0, B, 1, B)], 1, dests=[]),                     # one destination per region
                S.Chunk([(0, B, 1, B)], 1, peers=0b100)):                 # a rank outside the plan
        with pytest.raises(S.PlanError) as e:
            plan_of([S.Schedule([bad]), S.Schedule()])
        assert e.value.code == "EINVAL"


def test_groups_with_chunks_for_some_peers():
    # a group counts, at each rank, only the members that reach it (its own, or addressed to
    # it); the wait passes exactly when those are readable there, at every step of random orders
    rng = np.random.default_rng(12)
    P, B = 4, 8
    plan = _reduce_scatter_plan(P, B)
    groups = [[c for c in range(plan.G) if plan.chunks[c].receivers(P, plan.owner[c]) == [b]]
              for b in range(P)] + [list(range(plan.G))]
    plan.define_groups(groups)
    for R in (1, 2):
        plan.start()
        marks = [(r, c) for r in range(P) for c in plan.chunks_of(r)]
        for i in rng.permutation(len(marks)):
            plan.mark_ready(*marks[i])
            if rng.random() < 0.5:
                plan.copier_progress()
            for q in range(P):
                for g, members in enumerate(groups):
                    want = all(plan.chunk_readable(q, c) for c in members if plan.reaches(q, c))
                    assert plan.group_ready(q, g) == want
        plan.copier_progress()
        assert plan.wait()[0] == PL.OK
        for q in range(P):
            assert int(plan.group_counters[q, q]) == R * (P - 1)         # its P - 1 partials
        plan.next_round()
