"""GPU: the copier launched early for the next round (opts.early_copier_us) against the oracle.

dtt_plan_wait launches round R+1's copier behind round R's; dtt_plan_start(R+1) claims it through
a compare-and-swap on a mapped host word, or, when it has already given the round up, launches a
fresh one.  Whatever happens, every round's buffers and gate words must equal the oracle's: a
round is copied exactly once (an extra arrival would open a later round's wait early).
"""
import time

import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import assert_buffers_equal, oracle_plan, oracle_round
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner


def _opts(us, **kw):
    return D.dtt_plan_opts_default(early_copier_us=us, **kw)


def _check_round(st, o, w, R):
    assert oracle_round(o, w) == (OP.OK, [], [])
    for q in range(w.P):
        np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"round {R} buffer {q}")
    np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)


CASES = {
    "chunks_vector": (W.small(W.C2, M=96, N=512, num_chunks=6), {}),
    "chunks_bulk_group": (W.small(W.C2, M=96, N=1024, num_chunks=6),
                          {"group": 3, "programs": 2, "opts": dict(method=1, piece_bytes=16384, stages=4)}),
    "tiles_bulk_paced": (W.Workload("tp", P=4, M=512, N=512, dtype=W.BF16, kind="tile_chunks", rounds=4,
                                    seed=16, BM=64, BN=64, num_programs=6, tiles_per_chunk=6, group_m=3),
                         {"pace": 2, "threads": 128,
                          "opts": dict(method=1, piece_bytes=8192, stages=2, ctas_per_sm=3)}),
    "whole_after_producer": (W.small(W.C4A, M=64, N=64, rounds=4),
                             {"opts": dict(method=1, piece_bytes=4096, stages=2, deferred_copier=2)}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_early_copier_rounds_match_the_oracle(name):
    # a generous wait (1 s) so that the checks between rounds never outlast it: every round after
    # the first is copied by the copier launched in the previous wait
    w, kw = CASES[name]
    kw = dict(kw)
    st = runner.make(w, opts=_opts(1000000, **kw.pop("opts", {})), **kw)
    o = oracle_plan(w)
    rounds = 4
    try:
        for R in range(1, rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            _check_round(st, o, w, R)
            st.plan.next_round()
            o.next_round()
        e = st.plan.early_stats()
        assert e["launched"] == rounds and e["claimed"] == rounds - 1, e
        assert e["expired"] == 0 and e["aborted"] == 0, e
    finally:
        t0 = time.perf_counter()
        st.plan.close()                  # aborts the copier launched for round rounds + 1
        assert time.perf_counter() - t0 < 0.5
    assert st.plan.state == D.CLOSED


def test_early_copier_that_expired_is_replaced():
    # the host takes longer than the early copier waits: it gives its round up, start() finds
    # that and launches a fresh copier; the round is still copied exactly once
    w = W.small(W.C2, M=64, N=512, num_chunks=4)
    st = runner.make(w, opts=_opts(200))
    o = oracle_plan(w)
    try:
        for R in range(1, 5):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            _check_round(st, o, w, R)
            time.sleep(0.02)             # 20 ms >> 200 us
            st.plan.next_round()
            o.next_round()
        e = st.plan.early_stats()
        assert e["launched"] == 4 and e["expired"] == 3 and e["claimed"] == 0, e
    finally:
        st.plan.close()


def test_close_aborts_a_pending_early_copier_at_once():
    w = W.small(W.C2, M=64, N=512, num_chunks=4)
    for advance in (False, True):        # closed DONE, or PREPARED after next_round
        st = runner.make(w, opts=_opts(1000000))
        rep = runner.run_round(st)
        assert rep.status == D.OK
        if advance:
            st.plan.next_round()
        t0 = time.perf_counter()
        st.plan.close()
        assert time.perf_counter() - t0 < 0.5       # not the 1 s the early copier would wait
        assert st.plan.state == D.CLOSED


def test_failed_round_aborts_the_early_copier():
    # one chunk short of its marks: wait reports ETIMEDOUT, the copier launched for the next
    # round is aborted, and close returns at once
    w = W.small(W.C2, M=64, N=512, num_chunks=4)
    st = runner.make(w, opts=_opts(1000000, max_polls=1 << 14))
    try:
        h = st.plan.start(st.producer_stream)
        n_global, first, n_chunks, _ = st.plan.info()
        D.dtt_publish(h, 0, n_global - 1, 0, st.producer_stream)      # the last chunk never opens
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.ETIMEDOUT and rep.shorts == [n_global - 1]
        e = st.plan.early_stats()
        assert e["launched"] == 1 and e["aborted"] == 1, e
    finally:
        t0 = time.perf_counter()
        st.plan.close()
        assert time.perf_counter() - t0 < 0.5


def test_host_buffer_round_replaces_the_early_copier():
    # dtt_allgather_host needs a copier that stamps arrivals for the host: a pending early copier
    # is aborted and a stamping one launched; results equal the closed form
    w = W.small(W.C2, M=128, N=1024, num_chunks=4)
    st = runner.make(w, opts=_opts(1000000))
    S = w.slice_bytes
    try:
        assert runner.run_round(st).status == D.OK          # leaves an early copier pending
        st.plan.next_round()
        for R in (2, 3):
            host = [torch.from_numpy(np.full(S, 10 * R + r, dtype=np.uint8)).pin_memory() for r in range(w.P)]
            out = torch.empty(w.buf_bytes, dtype=torch.uint8).pin_memory()
            rep = st.plan.allgather_host(host, out, 1, st.producer_stream)
            assert rep.status == D.OK
            want = np.concatenate([np.full(S, 10 * R + r, dtype=np.uint8) for r in range(w.P)])
            np.testing.assert_array_equal(out.numpy(), want)
        e = st.plan.early_stats()
        assert e["launched"] == 1 and e["aborted"] == 1, e
        assert runner.run_round(st).status == D.OK          # an ordinary round after them
    finally:
        st.plan.close()


def test_shared_copy_stream_launches_at_start():
    # two plans on one copy stream: a copier launched early would hold the stream until its
    # plan's next start, so neither plan launches early; both stay correct
    w = W.small(W.C2, M=64, N=512, num_chunks=4)
    cs = torch.cuda.Stream()
    a = runner.make(w, opts=_opts(1000000), copy_stream=cs)
    b = runner.make(w, opts=_opts(1000000), copy_stream=cs)
    oa, ob = oracle_plan(w), oracle_plan(w)
    try:
        for R in (1, 2):
            for st, o in ((a, oa), (b, ob)):
                assert runner.run_round(st).status == D.OK
                _check_round(st, o, w, R)
                st.plan.next_round()
                o.next_round()
        assert a.plan.early_stats()["launched"] == 0 and b.plan.early_stats()["launched"] == 0
    finally:
        a.plan.close()
        b.plan.close()


def test_early_copier_c2_full_size_bench_launch():
    # the benchmark's c2 launch with the early copier: every byte of every buffer, every round.
    # The oracle's buffers are computed before the rounds, so that the work between two rounds
    # stays well inside the early copier's wait.
    from oracle import cfill
    w = W.C2
    launch = dict(runner.bench_launch(w, overlap=False))     # rounds one at a time
    launch["opts"].early_copier_us = 1000000
    want = [cfill.expected_buffer(w, R) for R in range(1, w.rounds + 1)]
    # load the comparison's kernels now: with lazy module loading a kernel's first launch waits
    # for the device to go idle, which a waiting early copier delays until it gives up
    x = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert_buffers_equal([x], x.clone(), "warm-up")
    (x != x).nonzero()
    torch.cuda.synchronize()
    st = runner.make(w, **launch)
    o = oracle_plan(w, copy_data=False)
    try:
        for R in range(1, w.rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w)[0] == OP.OK
            assert_buffers_equal(st.bufs, torch.from_numpy(want[R - 1]).cuda(), f"round {R}")
            np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
            st.plan.next_round()
            o.next_round()
        e = st.plan.early_stats()
        assert e["claimed"] + e["expired"] == w.rounds - 1 and e["claimed"] >= w.rounds - 2, e
    finally:
        st.plan.close()
