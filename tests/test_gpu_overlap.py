"""GPU: overlapping rounds (opts.overlap) against the oracle's overlapped plan.

"Triggered Plans", Not supported yet: "Overlapping rounds" -- wait() had to return before
next_round() could prepare the next round.  The oracle (oracle/plan.py, ``overlap=True``) reads
the feature as at most two rounds in flight: next_round() from RUNNING leaves the round pending,
each (source, peer) queue serves the pending round first, round R's producer writes a chunk only
once round R-1's copies of it have landed, and wait() reports the pending round first, taking
extra marks from the error word alone.  These tests drive the library and the oracle through the
same host calls and compare every buffer byte and gate word, the reports of every wait, a
snapshot taken between two rounds in flight (no copy may carry the next round's bytes), and the
hand-worked check cases of the oracle's own pins.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import assert_buffers_equal, expected_on_device
from oracle import gemm as OG
from oracle import hashfill as H
from oracle import plan as OP
from oracle import run as OR

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner


# ---- the oracle through the same host calls -------------------------------------------------

def _oracle_plan(w, copy_data=True, initial_round=1):
    n = w.buf_bytes if copy_data else 1
    bufs = [np.zeros(n, dtype=np.uint8) for _ in range(w.P)]
    return OP.Plan(bufs, OR.schedules(w), allgather=not w.broadcast, initial_round=initial_round,
                   validate=copy_data, copy_data=copy_data, overlap=True)


def _round_data(w, r, R):
    d = np.zeros(w.buf_bytes, dtype=np.uint8)
    off = w.slice_offset(r)
    d[off:off + w.slice_bytes] = H.fill_slice_bytes(w.dtype, w.seed, r, R, w.M, w.N)
    return d


def _oracle_produce(o, w, R):
    """Round R's producers: each chunk written once it is writable (the copier steps until it
    is), then marked by its writers."""
    for r in w.senders():
        data = _round_data(w, r, R) if o.copy_data else None
        for c in o.chunks_of(r):
            while not o.writable(r, c, R):
                assert o.copier_progress() > 0
            if data is not None:
                o.write_chunk(r, c, data, R)
            for _ in range(o.chunks[c].writers):
                o.mark_ready(r, c, R)


def _oracle_overlapped(w, rounds, copy_data=True):
    """runner.run_overlapped's host sequence on the oracle; returns the plan and each wait's
    (status, short, extra) in round order."""
    o = _oracle_plan(w, copy_data)
    results = []
    for i in range(rounds):
        R = o.start()
        _oracle_produce(o, w, R)
        if o.pending is not None:
            o.copier_progress()
            results.append(o.wait())
        if i + 1 < rounds:
            o.next_round()
    o.copier_progress()
    results.append(o.wait())
    return o, results


def _opts(**kw):
    kw.setdefault("overlap", 1)
    return D.dtt_plan_opts_default(**kw)


def _check_reports(reps, results, rounds):
    assert [r.round for r in reps] == list(range(1, rounds + 1))
    assert all(r.status == D.OK and r.copier_timeouts == 0 and r.device_status == 0 for r in reps)
    assert results == [(OP.OK, [], [])] * rounds


# ---- overlapped rounds end to end -------------------------------------------------------------

CASES = {
    # the chunked benchmark launch: bulk copies, each rank's program a group of CTAs
    "chunks_bulk_group": (W.small(W.C2, M=256, N=1024, num_chunks=4, rounds=5), "bench", {}),
    "chunks_vec_ragged": (W.small(W.C2, M=70, N=256, num_chunks=8, rounds=4), None, {}),
    # a copier of one CTA per source: the next round's producer waits on it chunk by chunk
    "chunks_slow_copier": (W.small(W.C2, M=256, N=1024, num_chunks=8, rounds=4), None,
                           {"opts": dict(copier_ctas=4, copier_threads=32)}),
    "tiles_paced_bulk": (W.Workload("tp", P=4, M=512, N=512, dtype=W.BF16, kind="tile_chunks",
                                    rounds=4, seed=16, BM=64, BN=64, num_programs=6,
                                    tiles_per_chunk=6, group_m=3),
                         None, {"pace": 2, "threads": 128,
                                "opts": dict(method=1, piece_bytes=8192, stages=2, ctas_per_sm=3)}),
    "tiles_cluster2": (W.Workload("t2", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                  rounds=4, seed=10, BM=64, BN=48, num_programs=5,
                                  tiles_per_chunk=5, group_m=2), None, {"cluster": 2}),
    "whole_f32_8writers": (W.small(W.C4A, M=64, N=64, rounds=4), None, {}),
    "whole_group4_bulk": (W.small(W.C4A, M=64, N=64, rounds=4), None,
                          {"group": 4, "opts": dict(method=1, piece_bytes=4096, stages=4)}),
    "bcast_u8": (W.Workload("b", P=4, M=64, N=4096, dtype=W.U8, kind="whole", rounds=3, seed=9,
                            num_programs=8, broadcast=True), None, {}),
    # the copier launched by next_round (and by the last wait) rather than at start
    "deferred2": (W.small(W.C2, M=128, N=512, num_chunks=4, rounds=4), None,
                  {"opts": dict(deferred_copier=2)}),
    # the copy-engine transport: the proxy thread takes the next round behind the pending one
    "ce_chunks": (W.small(W.C2, M=70, N=256, num_chunks=8, rounds=4), None, {"opts": dict(method=2)}),
    "ce_tiles": (W.Workload("ct", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks", rounds=3,
                            seed=7, BM=64, BN=48, num_programs=5, tiles_per_chunk=5, group_m=2),
                 None, {"opts": dict(method=2)}),
    "single_rank": (W.Workload("s1", P=1, M=64, N=256, dtype=W.BF16, kind="chunks", rounds=3,
                               seed=21, num_chunks=4), None, {}),
}


def _launch(w, base, kw):
    launch = dict(runner.bench_launch(w)) if base == "bench" else {}
    kw = dict(kw)
    opts = kw.pop("opts", None)
    launch.update(kw)
    if base == "bench":
        o = launch["opts"]
        o.overlap = 1
        o.early_copier_us = 0
        if opts:
            for k, v in opts.items():
                setattr(o, k, v)
    else:
        launch["opts"] = _opts(**(opts or {}))
    return launch


@pytest.mark.parametrize("name", sorted(CASES))
def test_overlapped_rounds_match_the_oracle(name):
    w, base, kw = CASES[name]
    st = runner.make(w, **_launch(w, base, kw))
    try:
        reps = runner.run_overlapped(st, w.rounds)
        o, results = _oracle_overlapped(w, w.rounds)
        _check_reports(reps, results, w.rounds)
        assert st.plan.state == D.DONE and st.plan.pending == 0 and st.plan.round == w.rounds
        for q in range(w.P):
            np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"buffer {q}")
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
        # the plan goes on with rounds one at a time as well
        st.plan.next_round()
        assert runner.run_round(st).status == D.OK
    finally:
        st.plan.close()


def test_snapshot_between_two_rounds_in_flight():
    # Round 2's producer runs while round 1's slow copier (one 32-thread CTA per source) still
    # copies; round 2's copier is launched only by the last wait.  Right after round 1's wait,
    # every peer copy must hold round 1's bytes (none of round 2's: no torn copy) while each
    # rank's own rows hold round 2's -- the oracle's buffers at the same point -- and every
    # chunk's round-2 gate opened after its last round-1 arrival (the writable rule).
    w = W.small(W.C2, M=256, N=1024, num_chunks=8, rounds=3)
    st = runner.make(w, opts=_opts(copier_ctas=w.P, copier_threads=32, deferred_copier=2))
    o = _oracle_plan(w)
    try:
        for R in (1, 2):
            h = st.plan.start(st.producer_stream)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            assert o.start() == R
            if R == 1:
                _oracle_produce(o, w, 1)
                st.plan.next_round()
                o.next_round()
        # the oracle: round 1's copies first (round 2's writes wait for them), then round 2's
        _oracle_produce(o, w, 2)
        o.copier_progress()
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == 1
        assert o.wait() == (OP.OK, [], [])
        st.producer_stream.synchronize()
        assert st.plan.state == D.RUNNING and st.plan.pending == 0
        # the oracle has delivered round 2 too by now (its queues ran on); compare the state the
        # GPU holds -- round 1's copies, round 2's own rows -- with the closed forms instead
        S = w.slice_bytes
        for q in range(w.P):
            got = st.bufs[q].cpu().numpy()
            for r in range(w.P):
                want = H.fill_slice_bytes(w.dtype, w.seed, r, 2 if r == q else 1, w.M, w.N)
                np.testing.assert_array_equal(got[r * S:(r + 1) * S], want, err_msg=f"buffer {q} slice {r}")
        g = st.plan.read_gates()
        n_global, first, n_chunks, _ = st.plan.info()
        t_open, t_arr = g[:, :, D.GATE_T_OPEN].astype(np.int64), g[:, :, D.GATE_T_ARRIVE].astype(np.int64)
        overlapped = False
        last_arrival = max(int(t_arr[q, c]) for s in range(w.P) for c in range(first[s], first[s] + n_chunks[s])
                           for q in range(w.P) if q != s)
        for s in range(w.P):
            for c in range(first[s], first[s] + n_chunks[s]):
                assert int(g[s, c, D.GATE_READY]) == 2
                arrivals = [int(t_arr[q, c]) for q in range(w.P) if q != s]
                assert int(t_open[s, c]) >= max(arrivals), (s, c)
                overlapped |= int(t_open[s, c]) < last_arrival
        assert overlapped, "round 2's producer did not run while round 1's copier was copying"
        rep = st.plan.wait()                  # round 2: its copier runs now
        assert rep.status == D.OK and rep.round == 2
        assert_buffers_equal(st.bufs, expected_on_device(w, 2), "round 2")
        np.testing.assert_array_equal(g[:, :, D.GATE_COUNTER], o.gates[:, :, OP.COUNTER])
    finally:
        st.plan.close()


def test_full_size_c2_bench_launch_overlapped():
    # the benchmark's c2 launch with overlapping rounds: every byte of every buffer after the
    # last round, and the gates, against the oracle
    w = W.C2
    st = runner.make(w, **_launch(w, "bench", {}))
    try:
        reps = runner.run_overlapped(st, w.rounds)
        o, results = _oracle_overlapped(w, w.rounds, copy_data=False)
        _check_reports(reps, results, w.rounds)
        assert_buffers_equal(st.bufs, expected_on_device(w, w.rounds), "c2 overlapped")
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


def test_full_size_c3_bench_launch_overlapped():
    w = W.C3
    rounds = 3
    st = runner.make(w, **_launch(w, "bench", {}))
    try:
        reps = runner.run_overlapped(st, rounds)
        o, results = _oracle_overlapped(w, rounds, copy_data=False)
        _check_reports(reps, results, rounds)
        assert_buffers_equal(st.bufs, expected_on_device(w, rounds), "c3 overlapped")
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


# ---- the GEMM producer ----------------------------------------------------------------------

def test_gemm_producer_overlapped_rounds_alternate_inputs():
    # Rounds alternate between two A operands, so a copy that carried the next round's C would
    # be off by the difference of two random products.  After round 1's wait (round 2's GEMM
    # done, its copier not yet launched), every peer copy of C_r is round 1's and every rank's
    # own C_r is round 2's; after the last round every copy equals its rank's C bit for bit.
    w5 = W.small(W.C5, M=256, N=512, K=256, num_programs=8, tiles_per_chunk=8)
    A0, Bt = W.gemm_inputs(w5.P, w5.M, w5.N, w5.K, w5.seed)
    A1, _ = W.gemm_inputs(w5.P, w5.M, w5.N, w5.K, w5.seed + 1)
    st = runner.make_gemm(w5, A0, Bt, opts=_opts(method=D.COPY_VEC16, deferred_copier=2))
    As = [st.A, A1.to("cuda").contiguous()]
    Bt64 = Bt.to(torch.float64).numpy()
    ref = [[OG.product(A[r].to(torch.float64).numpy(), Bt64) for r in range(w5.P)] for A in (A0, A1)]
    S = w5.M * w5.row_bytes

    def c_of(q, r):
        return st.bufs[q][r * S:(r + 1) * S].view(torch.bfloat16).view(w5.M, w5.N)

    def produce(R, handles):
        D.dtt_gemm_producer(As[(R - 1) % 2], st.Bt, st.buf_ptrs, w5.M, w5.N, w5.K, w5.row_bytes,
                            st.slice_offs, st.num_programs, handles, st.err, st.producer_stream)

    rounds = 4
    o = _oracle_plan(w5, copy_data=False)
    try:
        for R in range(1, rounds + 1):
            produce(R, st.plan.start(st.producer_stream))
            assert o.start() == R
            _oracle_produce(o, w5, R)
            if st.plan.pending:
                o.copier_progress()
                assert o.wait() == (OP.OK, [], [])
                rep = st.plan.wait()
                assert rep.status == D.OK and rep.round == R - 1 and int(st.err.item()) == 0
                if R == 2:
                    st.producer_stream.synchronize()
                    for r in range(w5.P):
                        own = c_of(r, r).to(torch.float64).cpu().numpy()
                        assert OG.rel_frobenius(own, ref[1][r]) <= 1e-2, ("own", r)
                        for q in range(w5.P):
                            if q != r:
                                got = c_of(q, r).to(torch.float64).cpu().numpy()
                                assert OG.rel_frobenius(got, ref[0][r]) <= 1e-2, ("copy", q, r)
            if R < rounds:
                st.plan.next_round()
                o.next_round()
        rep = st.plan.wait()
        o.copier_progress()
        assert o.wait() == (OP.OK, [], [])
        assert rep.status == D.OK and rep.round == rounds and int(st.err.item()) == 0
        for r in range(w5.P):
            mine = c_of(r, r)
            assert OG.rel_frobenius(mine.to(torch.float64).cpu().numpy(), ref[(rounds - 1) % 2][r]) <= 1e-2
            for q in range(w5.P):
                assert torch.equal(c_of(q, r).view(torch.int16), mine.view(torch.int16)), (q, r)
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


# ---- the check while the next round counts (the oracle's hand-worked cases) -------------------

def _marks_plan(**kw):
    """Two ranks of two one-writer chunks each; a producer that only marks (dtt_publish)."""
    w = W.small(W.C2, P=2, M=64, N=256, num_chunks=2, rounds=2)
    st = runner.make(w, opts=_opts(**kw))
    return w, st


def _publish(st, handles, chunks, marks=1):
    for c in chunks:
        D.dtt_publish(handles, c, 1, marks, st.producer_stream)


def test_extra_mark_is_reported_by_its_rounds_wait():
    w, st = _marks_plan()
    o = _oracle_plan(w, copy_data=False)
    try:
        h = st.plan.start(st.producer_stream)
        _publish(st, h, [0, 1, 2, 3])
        _publish(st, h, [0])                  # chunk 0: a second mark for one writer
        st.plan.next_round()
        st.plan.start(st.producer_stream)
        o.start()
        for c in range(4):
            o.mark_ready(o.owner[c], c)
        o.mark_ready(0, 0)
        o.next_round()
        o.start()
        o.copier_progress()
        assert o.wait() == (OP.EXTRA, [], [0])
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.EEXTRA and rep.round == 1 and rep.extras == [0]
        assert st.plan.state == D.FAILED
    finally:
        st.plan.close()


def test_next_rounds_marks_are_not_extra_marks():
    w, st = _marks_plan()
    o = _oracle_plan(w, copy_data=False)
    try:
        h = st.plan.start(st.producer_stream)
        _publish(st, h, [0, 1, 2, 3])
        st.plan.next_round()
        h = st.plan.start(st.producer_stream)
        _publish(st, h, [1])                  # round 2's mark of chunk 1 before round 1's check
        st.producer_stream.synchronize()
        o.start()
        for c in range(4):
            o.mark_ready(o.owner[c], c)
        o.next_round()
        o.start()
        o.copier_progress()
        o.mark_ready(0, 1)
        assert o.wait() == (OP.OK, [], [])
        g = st.plan.read_gates()
        assert int(g[0, 1, D.GATE_COUNTER]) == 2 and int(g[0, 1, D.GATE_READY]) == 2
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == 1
        assert st.plan.state == D.RUNNING and st.plan.pending == 0
        _publish(st, h, [0, 2, 3])
        for c in (0, 2, 3):
            o.mark_ready(o.owner[c], c)
        o.copier_progress()
        assert o.wait() == (OP.OK, [], [])
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == 2 and st.plan.state == D.DONE
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


def test_missing_mark_is_short_in_the_pending_rounds_wait():
    w, st = _marks_plan(max_polls=1 << 12)
    o = _oracle_plan(w, copy_data=False)
    try:
        h = st.plan.start(st.producer_stream)
        _publish(st, h, [0, 2, 3])            # chunk 1 never marked
        st.plan.next_round()
        st.plan.start(st.producer_stream)
        o.start()
        for c in (0, 2, 3):
            o.mark_ready(o.owner[c], c)
        o.next_round()
        o.start()
        o.copier_progress()
        assert not o.writable(0, 1) and o.writable(0, 0)
        assert o.wait() == (OP.TIMEOUT, [1], [])
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.ETIMEDOUT and rep.round == 1 and rep.shorts == [1]
        assert st.plan.state == D.FAILED
    finally:
        st.plan.close()            # round 2 is still running: its gates are opened, copies drained


def test_overlap_state_rules():
    w, st = _marks_plan()
    try:
        h = st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:
            st.plan.define_groups([[0, 1]])   # a next-round arrival would count in this round's wait
        assert e.value.code == D.EINVAL
        _publish(st, h, [0, 1, 2, 3])
        st.plan.next_round()
        assert st.plan.pending == 1 and st.plan.round == 2 and st.plan.state == D.PREPARED
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()              # PREPARED, with round 1 in flight
        assert e.value.code == D.ESTATE
        with pytest.raises(D.DttError) as e:
            st.plan.allgather_host([None] * w.P)
        assert e.value.code == D.ESTATE
        h = st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()              # two rounds in flight already
        assert e.value.code == D.ESTATE
        _publish(st, h, [0, 1])               # round 2 half marked: close sends it as it stands
    finally:
        assert st.plan.close() == D.OK        # two rounds in flight: both drained
    seq = runner.make(w)                       # without overlap: next_round only from DONE
    try:
        h = seq.plan.start(seq.producer_stream)
        with pytest.raises(D.DttError) as e:
            seq.plan.next_round()
        assert e.value.code == D.ESTATE
        _publish(seq, h, [0, 1, 2, 3])
        assert seq.plan.wait().status == D.OK
    finally:
        seq.plan.close()


def test_overlapped_round_limit():
    # rounds 2^32 - 2 and 2^32 - 1 in flight together; no round follows them
    w = W.small(W.C2, P=2, M=64, N=256, num_chunks=2, rounds=2)
    first = (1 << 32) - 2
    st = runner.make(w, opts=_opts(initial_round=first))
    o = _oracle_plan(w, initial_round=first)
    try:
        for R in (first, first + 1):
            h = st.plan.start(st.producer_stream)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            assert o.start() == R
            _oracle_produce(o, w, R)
            if R == first:
                st.plan.next_round()
                o.next_round()
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()              # two rounds in flight
        assert e.value.code == D.ESTATE
        with pytest.raises(OP.StateError):
            o.next_round()
        o.copier_progress()
        assert o.wait() == (OP.OK, [], [])
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == first
        assert st.plan.state == D.RUNNING and st.plan.pending == 0
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()              # round 2^32 - 1 cannot leave a next round behind it
        assert e.value.code == D.EROUNDLIMIT
        assert st.plan.state == D.RUNNING and st.plan.pending == 0
        with pytest.raises(OP.RoundLimitError):
            o.next_round()
        assert o.wait() == (OP.OK, [], [])
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == first + 1
        for q in range(w.P):
            np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q])
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


def test_overlap_refuses_producer_ctas_larger_than_half_an_sm():
    # the next round's copier may take an SM before the next round's producer: a fill CTA of
    # 1024 threads could then never start beside it, so such a launch is refused up front
    w = W.small(W.C2, P=2, M=64, N=256, num_chunks=2, rounds=1)
    st = runner.make(w, opts=_opts(), threads=1024)
    try:
        h = st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        assert e.value.code == D.EINVAL
        st.desc.threads = 512
        D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        assert st.plan.wait().status == D.OK
    finally:
        st.plan.close()


def test_consumers_on_overlapped_rounds():
    # Each round's consumers -- the tcgen05 consumer GEMM and the gather, both waiting per chunk
    # -- run on a stream of their own, launched before the round's producer; the next round's
    # producer is ordered after them (whoever reads a round is done before the next round's
    # producers run), while the round's copier and check still overlap the next round.  Every
    # round's gathered bytes and product are checked against the oracle's closed form.
    w = W.small(W.C2, M=512, N=1024, num_chunks=4, rounds=4)
    K, N2, q = w.N, 256, 2
    rows = w.buf_bytes // (2 * K)
    g = torch.Generator().manual_seed(91)
    Wt = (torch.randn(N2, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    Wt_dev = Wt.cuda()
    Wt64 = Wt.to(torch.float64).numpy()
    st = runner.make(w, opts=_opts())
    n_global = st.plan.info()[0]
    cons = torch.cuda.Stream()
    outs = [torch.zeros(rows, N2, dtype=torch.bfloat16, device="cuda") for _ in range(w.rounds)]
    gath = [torch.zeros(w.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(w.rounds)]
    status = [torch.full((n_global,), 99, dtype=torch.int32, device="cuda") for _ in range(w.rounds)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    readers_done = None
    try:
        for i in range(w.rounds):
            h = st.plan.start(st.producer_stream)
            st.plan.gemm_consumer(q, Wt_dev, outs[i], N2, K, err, stream=cons)
            st.plan.consumer_gather(q, gath[i], 1 << 24, status[i], 8, cons)
            if readers_done is not None:
                st.producer_stream.wait_event(readers_done)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            readers_done = torch.cuda.Event()
            readers_done.record(cons)
            if st.plan.pending:
                rep = st.plan.wait()
                assert rep.status == D.OK and rep.round == i
            if i + 1 < w.rounds:
                st.plan.next_round()
        rep = st.plan.wait()
        assert rep.status == D.OK and rep.round == w.rounds
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        S = w.slice_bytes
        for i in range(w.rounds):
            want = OP.expected_allgather(w.P, w.M, w.N, w.dtype, w.seed, i + 1, w.elem_bytes)
            assert status[i].cpu().tolist() == [0] * n_global, i
            got = gath[i].cpu().numpy()
            for r in range(w.P):
                sl = slice(r * S, (r + 1) * S)
                np.testing.assert_array_equal(got[sl], want[sl] if r != q else 0, err_msg=f"round {i + 1} slice {r}")
            X = torch.from_numpy(want.copy()).view(torch.bfloat16).view(rows, K)
            e = OG.rel_frobenius(outs[i].cpu().to(torch.float64).numpy(), OG.product(X.to(torch.float64).numpy(), Wt64))
            assert e <= 1e-2, (i + 1, e)
    finally:
        st.plan.close()


def test_many_overlapped_rounds_keep_the_gates_and_data_right():
    # 500 rounds of the benchmark's c2 launch two at a time: every wait reports its own round,
    # the gates follow the closed form of the round count, and the data is the last round's
    # everywhere (every byte)
    w = W.C2
    R = 500
    st = runner.make(w, **_launch(w, "bench", {}))
    try:
        reps = runner.run_overlapped(st, R)
        assert [r.round for r in reps] == list(range(1, R + 1))
        assert all(r.status == D.OK and r.copier_timeouts == 0 for r in reps)
        g = st.plan.read_gates()
        n_global, first, n_chunks, _ = st.plan.info()
        for s in range(w.P):
            for c in range(first[s], first[s] + n_chunks[s]):
                assert int(g[s, c, D.GATE_READY]) == R and int(g[s, c, D.GATE_COUNTER]) == R
                assert int(g[s, c, D.GATE_COMPLETION]) == R * (w.P - 1)
                assert int(g[s, c, D.GATE_ERROR]) == 0
                for q in range(w.P):
                    if q != s:
                        assert int(g[q, c, D.GATE_ARRIVAL]) == R
        assert_buffers_equal(st.bufs, expected_on_device(w, R), f"{w.name} round {R}")
    finally:
        st.plan.close()


# ---- host-buffer rounds, pipelined across rounds ----------------------------------------------

HOST_ROUND_CASES = {
    "chunks_one_piece": (W.small(W.C2, M=128, N=512, num_chunks=4), {}),
    # 8 MiB slices go in as two 4 MiB pieces; 1 MiB chunks open as their bytes land
    "chunks_two_pieces_bulk": (W.small(W.C2, M=2048, N=2048, num_chunks=8),
                               {"opts": dict(method=1, piece_bytes=65536, stages=3)}),
    # 2D tile windows (tensor-map boxes), grouped order, slices of two pieces
    "tiles_two_pieces": (W.Workload("ht", P=3, M=3000, N=1024, dtype=W.BF16, kind="tile_chunks",
                                    rounds=2, seed=41, BM=128, BN=128, num_programs=6,
                                    tiles_per_chunk=6, group_m=4),
                         {"opts": dict(method=1, piece_bytes=16384, stages=12)}),
    # host copies of 12 KiB: many pieces per slice, chunk edges inside pieces
    "chunks_small_host_pieces": (W.small(W.C2, M=96, N=1024, num_chunks=6),
                                 {"opts": dict(host_piece_bytes=12288)}),
}


def _host_slices(w, R):
    """Round R's host slices: every round's values differ (a copy carrying another round's bytes
    shows), and the closed form of the gathered buffer is their concatenation."""
    return [torch.from_numpy(H.fill_slice_bytes(w.dtype, w.seed + R, r, R, w.M, w.N)).pin_memory()
            for r in range(w.P)]


@pytest.mark.parametrize("out_rank", ["first", "last"])
@pytest.mark.parametrize("name", sorted(HOST_ROUND_CASES))
def test_host_rounds_pipelined(name, out_rank):
    # rounds from and to host memory back to back, round k + 1's slices going in while round k's
    # gathered buffer comes back: every round's copy back is that round's concatenation
    w, kw = HOST_ROUND_CASES[name]
    q = 0 if out_rank == "first" else w.P - 1
    st = runner.make(w, opts=_opts(**kw.get("opts", {})))
    n = 5
    host = [_host_slices(w, R) for R in range(1, n + 1)]
    outs = [torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory() for _ in range(n)]
    try:
        reps = st.plan.allgather_host_rounds(host, outs, q, st.producer_stream)
        assert [r.round for r in reps] == list(range(1, n + 1))
        assert all(r.status == D.OK and r.copier_timeouts == 0 for r in reps)
        for k in range(n):
            want = np.concatenate([h.numpy() for h in host[k]])
            np.testing.assert_array_equal(outs[k].numpy(), want, err_msg=f"round {k + 1}")
        want = np.concatenate([h.numpy() for h in host[-1]])
        for b in st.bufs:
            np.testing.assert_array_equal(b.cpu().numpy(), want)
        assert st.plan.round == n + 1 and st.plan.state == D.PREPARED and st.plan.pending == 0
        # and one more round of the ordinary kind on the same plan
        more = _host_slices(w, n + 1)
        out = torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory()
        assert st.plan.allgather_host(more, out, q, st.producer_stream).status == D.OK
        np.testing.assert_array_equal(out.numpy(), np.concatenate([h.numpy() for h in more]))
    finally:
        st.plan.close()


def test_host_rounds_edges():
    # a round with a slice left as it stands, a round with no copy back, one round alone, and a
    # plan without overlapping rounds (refused)
    w = W.small(W.C2, M=1024, N=2048, num_chunks=4)
    S = w.slice_bytes
    st = runner.make(w, opts=_opts(), fill_byte=5)
    try:
        host = [_host_slices(w, R) for R in (1, 2, 3)]
        host[0][1] = None                       # round 1: rank 1's rows as they stand (5s)
        outs = [torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory() for _ in range(3)]
        outs[1] = None                          # round 2: nothing copied back
        reps = st.plan.allgather_host_rounds(host, outs, 0, st.producer_stream)
        assert [r.status for r in reps] == [D.OK] * 3
        want1 = np.concatenate([h.numpy() if h is not None else np.full(S, 5, np.uint8) for h in host[0]])
        np.testing.assert_array_equal(outs[0].numpy(), want1)
        np.testing.assert_array_equal(outs[2].numpy(), np.concatenate([h.numpy() for h in host[2]]))
        one = [_host_slices(w, 4)]
        out = [torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory()]
        rep = st.plan.allgather_host_rounds(one, out, w.P - 1, st.producer_stream)
        assert rep[0].status == D.OK and rep[0].round == 4
        np.testing.assert_array_equal(out[0].numpy(), np.concatenate([h.numpy() for h in one[0]]))
    finally:
        st.plan.close()
    seq = runner.make(w)
    try:
        with pytest.raises(D.DttError) as e:
            seq.plan.allgather_host_rounds([_host_slices(w, 1)], None, 0, seq.producer_stream)
        assert e.value.code == D.EINVAL
    finally:
        seq.plan.close()


def test_host_rounds_c2_full_size():
    # the benchmark's c2 launch from and to host memory, five rounds pipelined
    w = W.C2
    st = runner.make(w, **_launch(w, "bench", {}))
    n = 5
    host = [_host_slices(w, R) for R in range(1, n + 1)]
    outs = [torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory() for _ in range(n)]
    try:
        reps = st.plan.allgather_host_rounds(host, outs, 0, st.producer_stream)
        assert all(r.status == D.OK for r in reps)
        for k in range(n):
            want = torch.cat(host[k])
            assert torch.equal(outs[k], want), f"round {k + 1}"
    finally:
        st.plan.close()


@pytest.mark.parametrize("method", [0, 1, 2], ids=["vector", "bulk", "copy_engines"])
def test_overlap_close_and_wait_states(method):
    # close right after next_round (the next round PREPARED, this one pending), a second wait with
    # nothing left to check, and close with two rounds in flight on every transport
    w = W.small(W.C2, P=2, M=64, N=256, num_chunks=2, rounds=2)
    extra = dict(piece_bytes=16384, stages=2) if method == 1 else {}
    st = runner.make(w, opts=_opts(method=method, **extra))
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        st.plan.next_round()
        assert st.plan.state == D.PREPARED and st.plan.pending == 1
        rep = st.plan.wait()                  # round 1, with round 2 not started
        assert rep.status == D.OK and rep.round == 1
        assert st.plan.state == D.PREPARED and st.plan.pending == 0
        with pytest.raises(D.DttError) as e:
            st.plan.wait()                    # nothing running, nothing pending
        assert e.value.code == D.ESTATE
        want = OP.expected_allgather(w.P, w.M, w.N, w.dtype, w.seed, 1, w.elem_bytes)
        for q in range(w.P):
            np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), want)
        h = st.plan.start(st.producer_stream)
        D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        st.plan.next_round()                  # round 2 pending, round 3 PREPARED
    finally:
        assert st.plan.close() == D.OK        # the pending round drains
    st = runner.make(w, opts=_opts(method=method, **extra))
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        st.plan.next_round()
        st.plan.start(st.producer_stream)     # round 2 running with no producer: close opens it
    finally:
        assert st.plan.close() == D.OK


def test_overlap_with_copier_timing():
    # the copier timed by the library's events on overlapped rounds: one timed launch per round
    w = W.small(W.C2, M=128, N=512, num_chunks=4, rounds=6)
    st = runner.make(w, opts=_opts(time_copier=1))
    try:
        reps = runner.run_overlapped(st, w.rounds)
        assert [r.status for r in reps] == [D.OK] * w.rounds
        last, total, n = st.plan.stats()
        assert n == w.rounds and total >= last > 0
        want = OP.expected_allgather(w.P, w.M, w.N, w.dtype, w.seed, w.rounds, w.elem_bytes)
        for q in range(w.P):
            np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), want)
    finally:
        st.plan.close()
