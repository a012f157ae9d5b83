"""The triggered protocol with CPU threads as ranks (oracle/threaded.py)."""
import numpy as np
import pytest

from oracle import hashfill as H
from oracle import plan as PL
from oracle import schedule as S
from oracle.threaded import ThreadedRound, barrier_threads


def _setup(P=3, M=8, N=8, n=4):
    e = 2
    rb = N * e
    sb = M * rb
    bufs = [np.zeros(P * sb, dtype=np.uint8) for _ in range(P)]
    scheds = [S.chunks(r * sb, M, rb, rb, n) for r in range(P)]
    plan = PL.Plan(bufs, scheds)
    data = {r: H.fill_slice_bytes("bf16", 11, r, 1, M, N) for r in range(P)}

    def write_unit(rank, c, u):
        for (off, nb, rows, pitch) in plan.chunks[c].regions:
            lo = off - rank * sb
            plan.bufs[rank][off:off + nb] = data[rank][lo:lo + nb]

    order = {r: [(c, 0) for c in plan.chunks_of(r)] for r in range(P)}
    return plan, write_unit, order, data, sb


def test_threaded_round_matches_closed_form():
    plan, write_unit, order, data, sb = _setup()
    status = ThreadedRound(plan, write_unit, order, programs=2).run()
    assert status == (PL.OK, [], [])
    want = np.concatenate([data[r] for r in range(plan.P)])
    for q in range(plan.P):
        assert np.array_equal(plan.bufs[q], want)


def test_out_of_order_completion_is_correct_and_queues_keep_schedule_order():
    plan, write_unit, order, data, sb = _setup(P=2, n=4)
    for r in range(2):
        order[r] = list(reversed(order[r]))          # the producer completes chunks backwards
    delay = {(c, 0): 0.01 for c in range(plan.G)}
    tr = ThreadedRound(plan, write_unit, order, delay=delay)
    assert tr.run()[0] == PL.OK
    for (s, p), log in tr.queue_log.items():
        assert log == list(plan.chunks_of(s))        # head-of-line: schedule order per queue
    want = np.concatenate([data[r] for r in range(2)])
    assert all(np.array_equal(b, want) for b in plan.bufs)


def test_missing_mark_times_out_naming_the_chunk():
    plan, write_unit, order, data, sb = _setup(P=2, n=2)
    tr = ThreadedRound(plan, write_unit, order, max_polls=200, skip={(2, 0)})
    status, short, extra = tr.run()
    # chunk 2 never opens; chunk 3 opened but waits behind it on the same queue
    assert status == PL.TIMEOUT and short == [2, 3] and extra == []
    assert int(plan.gates[1, 3, PL.READY]) == 1 and int(plan.gates[0, 3, PL.ARRIVAL]) == 0
    assert (0, 1, 2) not in [(s, p, c) for (s, p, c) in tr.timeouts] and \
        any(c == 2 for (s, p, c) in tr.timeouts)


def test_extra_mark_reported():
    plan, write_unit, order, data, sb = _setup(P=2, n=2)
    status, short, extra = ThreadedRound(plan, write_unit, order, extra={(1, 0)}).run()
    assert status == PL.EXTRA and extra == [1]


def test_close_mid_round_drains():
    plan, write_unit, order, data, sb = _setup(P=2, n=2)
    tr = ThreadedRound(plan, write_unit, order, max_polls=100000, skip={(1, 0), (3, 0)})
    assert tr.run(close_after=0.05) is None
    assert plan.state == "CLOSED"
    # every chunk was delivered once; the gates of the unmarked chunks were opened by close
    assert all(int(plan.gates[p, c, PL.ARRIVAL]) == 1
               for c in range(plan.G) for p in range(2) if p != plan.owner[c])


@pytest.mark.parametrize("P", [2, 3, 8])
def test_barrier_threads(P):
    ys = barrier_threads(P, gen_calls=3)
    for r in range(P):
        want = np.full(P, 3)
        want[r] = 0
        assert np.array_equal(ys[r], want)


def test_group_waits_with_threads():
    # consumer threads wait once on a group (chunks of several source ranks, one of them the
    # consumer's own) and then read every chunk of it: the data is there; the producers complete
    # chunks backwards, so the groups open only at the end of each queue
    plan, write_unit, order, data, sb = _setup(P=3, n=4)
    groups = [[0, 5, 10], [1, 2, 3], list(range(plan.G)), [7]]
    plan.define_groups(groups)
    for r in range(3):
        order[r] = list(reversed(order[r]))
    waits = [(q, g) for q in range(3) for g in range(len(groups))]
    tr = ThreadedRound(plan, write_unit, order, delay={(c, 0): 0.003 for c in range(plan.G)},
                       group_waits=waits)
    assert tr.run()[0] == PL.OK
    assert all(tr.consumer_results[k] == "ok" for k in waits), tr.consumer_results
    for q in range(3):
        for g, members in enumerate(groups):
            assert int(plan.group_counters[q, g]) == len(members)


def test_group_wait_times_out_on_a_missing_mark():
    plan, write_unit, order, data, sb = _setup(P=2, n=2)
    plan.define_groups([[0, 3], [0, 1]])
    tr = ThreadedRound(plan, write_unit, order, max_polls=300, skip=[(3, 0)],
                       group_waits=[(0, 0), (1, 0), (0, 1), (1, 1)])
    status, short, extra = tr.run()
    assert status == PL.TIMEOUT and short == [3]
    assert tr.consumer_results[(0, 0)] == "timeout" and tr.consumer_results[(1, 0)] == "timeout"
    assert tr.consumer_results[(0, 1)] == "ok" and tr.consumer_results[(1, 1)] == "ok"


def test_reduce_scatter_with_threads_and_group_waits():
    # each rank sends partial block b only to rank b's staging slot; rank b's consumer waits once
    # on the group of its P - 1 incoming partials and then reads them all
    P, B = 3, 16
    bufs = [np.zeros(2 * P * B, dtype=np.uint8) for _ in range(P)]
    scheds = [S.Schedule([S.Chunk([(b * B, B, 1, B)], 1, dests=[(P * B + s * B, B)], peers=1 << b)
                          for b in range(P) if b != s]) for s in range(P)]
    plan = PL.Plan(bufs, scheds, allgather=False)
    groups = [[c for c in range(plan.G) if plan.chunks[c].peers == 1 << b] for b in range(P)]
    plan.define_groups(groups)
    data = {s: ((np.arange(P * B) * 3 + 17 * s) % 256).astype(np.uint8) for s in range(P)}

    def write_unit(rank, c, u):
        off, nb, _, _ = plan.chunks[c].regions[0]
        plan.bufs[rank][off:off + nb] = data[rank][off:off + nb]

    order = {r: [(c, 0) for c in reversed(list(plan.chunks_of(r)))] for r in range(P)}
    tr = ThreadedRound(plan, write_unit, order, group_waits=[(b, b) for b in range(P)],
                       delay={(c, 0): 0.002 for c in range(plan.G)})
    assert tr.run()[0] == PL.OK
    assert all(tr.consumer_results[(b, b)] == "ok" for b in range(P))
    for b in range(P):
        for s in range(P):
            if s != b:
                assert np.array_equal(plan.bufs[b][P * B + s * B:P * B + (s + 1) * B], data[s][b * B:(b + 1) * B])
