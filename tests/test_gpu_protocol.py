"""GPU: the plan's protocol edges -- extra and missing marks, the round limit, close in
mid-round, the consumer-side wait (and its timeout), state errors, the host-buffer round --
each against what the oracle says for the same sequence of events."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import oracle_plan, oracle_round
from oracle import hashfill as H
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner

WS = W.Workload("p", P=2, M=64, N=128, dtype=W.BF16, kind="chunks", rounds=3, seed=21,
                num_chunks=2)


def _fast_timeout_opts():
    return D.dtt_plan_opts_default(max_polls=20000)


def test_extra_mark_is_reported():
    st = runner.make(WS)
    o = oracle_plan(WS)
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_fill_producer(st.bufs, st.desc, h, st.producer_stream)
        D.dtt_publish(h, 1, 1, 1, st.producer_stream)           # one mark too many on chunk 1
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.EEXTRA and rep.extras == [1]
        assert st.plan.state == D.FAILED
        o.start()
        for r in range(2):
            off = WS.slice_offset(r)
            o.bufs[r][off:off + WS.slice_bytes] = H.fill_slice_bytes(WS.dtype, WS.seed, r, 1, WS.M, WS.N)
            for c in o.chunks_of(r):
                o.mark_ready(r, c)
        o.mark_ready(0, 1)
        o.copier_progress()
        assert o.wait() == (OP.EXTRA, [], [1])
        g = st.plan.read_gates()
        np.testing.assert_array_equal(g[:, :, :5], o.gates)
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()
        assert e.value.code == D.ESTATE
    finally:
        st.plan.close()


def test_missing_mark_times_out_and_names_short_chunks():
    st = runner.make(WS, opts=_fast_timeout_opts())
    o = oracle_plan(WS)
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_publish(h, 0, 2, 0, st.producer_stream)   # rank 0: both chunks
        D.dtt_publish(h, 3, 1, 0, st.producer_stream)   # rank 1: chunk 3 only; chunk 2 is short
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.ETIMEDOUT
        o.start()
        for c in (0, 1):
            o.mark_ready(0, c)
        o.mark_ready(1, 3)
        o.copier_progress()
        status, short, extra = o.wait()
        assert status == OP.TIMEOUT and rep.shorts == short == [2, 3]
        assert rep.copier_timeouts >= 1
        g = st.plan.read_gates()
        np.testing.assert_array_equal(g[:, :, :5], o.gates)
    finally:
        st.plan.close()


def test_round_limit():
    top = (1 << 32) - 1
    st = runner.make(WS, opts=D.dtt_plan_opts_default(initial_round=top - 1))
    o = oracle_plan(WS, initial_round=top - 1)
    try:
        for R in (top - 1, top):
            assert st.plan.round == R
            assert runner.run_round(st).status == D.OK
            assert oracle_round(o, WS)[0] == OP.OK
            np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
            for q in range(2):
                np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q])
            if R < top:
                st.plan.next_round()
                o.next_round()
        with pytest.raises(D.DttError) as e:
            st.plan.next_round()
        assert e.value.code == D.EROUNDLIMIT
        assert st.plan.state == D.DONE
    finally:
        st.plan.close()


def test_state_errors():
    st = runner.make(WS)
    try:
        for f in (st.plan.wait, st.plan.next_round):
            with pytest.raises(D.DttError) as e:
                f()
            assert e.value.code == D.ESTATE
        st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:
            st.plan.start(st.producer_stream)
        assert e.value.code == D.ESTATE
        D.dtt_fill_producer(st.bufs, st.desc, st.plan.handles, st.producer_stream)
        assert st.plan.wait().status == D.OK
    finally:
        st.plan.close()


def test_plan_without_chunks_runs_empty_rounds():
    # every schedule empty: no copier is launched, the check has nothing to report, and rounds
    # still advance one at a time
    P, S = 3, 4096
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_empty() for _ in range(P)]
    plan = D.Plan(bufs, P * S, scheds)
    for s in scheds:
        s.free()
    prod = torch.cuda.Stream()
    try:
        for R in (1, 2, 3):
            h = plan.start(prod)
            assert [h[r].n_chunks for r in range(P)] == [0] * P and h[0].round == R
            rep = plan.wait()
            assert rep.status == D.OK and rep.n_short == 0 and rep.n_extra == 0
            assert plan.next_round() == R + 1
    finally:
        plan.close()


@pytest.mark.parametrize("method", [0, 1])
def test_zero_byte_chunk_opens_and_arrives(method):
    # a chunk whose only region has no bytes still takes its writers' marks, opens, and arrives
    # at every peer in schedule order between its neighbours ("Triggered Plans", Gates and rounds)
    P, rows, rb = 3, 8, 256
    S = rows * rb
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = []
    for r in range(P):
        sc = D.dtt_schedule_empty()
        sc.add_chunk([(r * S, 4 * rb, 1, 4 * rb)], 1)
        sc.add_chunk([(r * S, 0, 1, 0)], 2)                    # zero bytes, two writers
        sc.add_chunk([(r * S + 4 * rb, 4 * rb, 1, 4 * rb)], 1)
        scheds.append(sc)
    plan = D.Plan(bufs, P * S, scheds, D.dtt_plan_opts_default(method=method, piece_bytes=512))
    for sc in scheds:
        sc.free()
    prod = torch.cuda.Stream()
    try:
        for R in (1, 2):
            h = plan.start(prod)
            want = torch.cat([torch.full((S,), 10 * R + r, dtype=torch.uint8) for r in range(P)])
            with torch.cuda.stream(prod):
                for r in range(P):
                    bufs[r][r * S:(r + 1) * S].copy_(want[r * S:(r + 1) * S].cuda(), non_blocking=False)
            D.dtt_publish(h, 0, 3 * P, 0, prod)        # every chunk: its writer count of marks
            rep = plan.wait()
            assert rep.status == D.OK
            for q in range(P):
                assert torch.equal(bufs[q].cpu(), want)
            g = plan.read_gates()
            for c in range(3 * P):
                owner = c // 3
                assert int(g[owner, c, D.GATE_READY]) == R
                assert int(g[owner, c, D.GATE_COMPLETION]) == R * (P - 1)
                for q in range(P):
                    if q != owner:
                        assert int(g[q, c, D.GATE_ARRIVAL]) == R
            plan.next_round()
    finally:
        plan.close()


def test_producer_stream_must_differ_from_copy_stream():
    copy = torch.cuda.Stream()
    bufs = [torch.zeros(WS.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    plan = D.Plan(bufs, WS.buf_bytes, runner.schedules_for(WS), copy_stream=copy)
    with pytest.raises(D.DttError) as e:
        plan.start(copy)
    assert e.value.code == D.EINVAL
    plan.close()


def test_copier_must_leave_room_for_the_producer():
    # a 1024-thread vector copier CTA on every SM would hold all of its registers while it spins,
    # so no producer CTA could run beside it: refused unless the copier is deferred
    bufs = [torch.zeros(WS.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    with pytest.raises(D.DttError) as e:
        D.Plan(bufs, WS.buf_bytes, runner.schedules_for(WS),
               D.dtt_plan_opts_default(copier_threads=1024))
    assert e.value.code == D.EINVAL
    st = runner.make(WS, opts=D.dtt_plan_opts_default(copier_threads=1024, deferred_copier=1))
    try:
        rep = runner.run_round(st)
        assert rep.status == D.OK
    finally:
        st.plan.close()


def test_bulk_copier_whose_rings_cannot_all_be_resident_is_refused():
    # four bulk-copy CTAs per SM with 2 x 32 KiB rings need more shared memory than an SM has: a
    # copier CTA waiting for room would keep the producer from starting, so creation refuses
    # it (unless the copier is deferred); three such CTAs fit
    bufs = [torch.zeros(WS.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    for cps, stages, piece in [(4, 2, 32768), (3, 3, 32768), (2, 2, 65536)]:
        with pytest.raises(D.DttError) as e:
            D.Plan(bufs, WS.buf_bytes, runner.schedules_for(WS),
                   D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=cps, stages=stages, piece_bytes=piece))
        assert e.value.code == D.EINVAL and "shared memory" in str(e.value)
    for opts in (D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=3, stages=2, piece_bytes=32768),
                 D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=4, stages=2, piece_bytes=32768,
                                         deferred_copier=1)):
        st = runner.make(WS, opts=opts)
        try:
            assert runner.run_round(st).status == D.OK
        finally:
            st.plan.close()


def test_bulk_copier_needs_two_stages():
    bufs = [torch.zeros(WS.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    with pytest.raises(D.DttError) as e:
        D.Plan(bufs, WS.buf_bytes, runner.schedules_for(WS),
               D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=65536, stages=1))
    assert e.value.code == D.EINVAL


def test_close_mid_round_sends_chunks_as_they_stand():
    st = runner.make(WS)
    o = oracle_plan(WS)
    # made before the round starts: a first-use kernel launched while the copier spins could
    # wait on it (lazy module loading)
    data = torch.arange(WS.slice_bytes, dtype=torch.int64).remainder(251).to(torch.uint8).cuda()
    st.producer_stream.wait_stream(torch.cuda.current_stream())
    h = st.plan.start(st.producer_stream)
    with torch.cuda.stream(st.producer_stream):
        st.bufs[0][:WS.slice_bytes // 2].copy_(data[:WS.slice_bytes // 2])
    D.dtt_publish(h, 0, 1, 0, st.producer_stream)       # rank 0 marks its first chunk only
    st.plan.close()                                      # opens every gate still closed
    torch.cuda.synchronize()
    o.start()
    o.bufs[0][:WS.slice_bytes // 2] = data[:WS.slice_bytes // 2].cpu().numpy()
    o.mark_ready(0, 0)
    o.close()
    for q in range(2):
        np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q])


def test_consumer_wait_reads_this_rounds_data():
    w = W.small(W.C2, M=256, N=1024, num_chunks=4)
    st = runner.make(w)
    o = oracle_plan(w)
    n_global = st.plan.info()[0]
    dst = torch.zeros(w.buf_bytes, dtype=torch.uint8, device="cuda")
    status = torch.full((n_global,), 99, dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        for R in (1, 2):
            h = st.plan.start(st.producer_stream)
            st.plan.consumer_gather(1, dst, 1 << 24, status, 4, cons)
            D.dtt_fill_producer(st.bufs, st.desc, h, st.producer_stream)
            st.plan.wait()
            cons.synchronize()
            assert oracle_round(o, w)[0] == OP.OK
            assert status.cpu().tolist() == [0] * n_global
            got = dst.cpu().numpy()
            S = w.slice_bytes
            for r in range(w.P):
                if r != 1:   # every other rank's slice, as this round left it
                    np.testing.assert_array_equal(got[r * S:(r + 1) * S], o.bufs[1][r * S:(r + 1) * S])
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


def test_consumer_wait_times_out_on_a_gate_nobody_opens():
    st = runner.make(WS, opts=_fast_timeout_opts())
    n_global = st.plan.info()[0]
    dst = torch.zeros(WS.buf_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros((n_global,), dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    torch.cuda.synchronize()
    st.plan.start(st.producer_stream)
    st.plan.consumer_gather(0, dst, 2000, status, 2, cons)   # no producer runs this round
    cons.synchronize()
    assert status.cpu().tolist() == [0, 0, D.ETIMEDOUT, D.ETIMEDOUT]
    st.plan.close()


HOST_CASES = {
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


@pytest.mark.parametrize("name", sorted(HOST_CASES))
def test_allgather_from_host_buffers(name):
    w, kw = HOST_CASES[name]
    kw = dict(kw)
    opts = kw.pop("opts", None)
    st = runner.make(w, opts=D.dtt_plan_opts_default(**opts) if opts else None)
    try:
        for R in (1, 2):
            host = [torch.from_numpy(H.fill_slice_bytes(w.dtype, w.seed + R, r, R, w.M, w.N)).pin_memory()
                    for r in range(w.P)]
            out = torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory()
            rep = st.plan.allgather_host(host, out, out_rank=w.P - 1, stream=st.producer_stream)
            assert rep.status == D.OK
            want = np.concatenate([h.numpy() for h in host])
            np.testing.assert_array_equal(out.numpy(), want)
            for q in range(w.P):
                np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), want)
        assert st.plan.round == 3
    finally:
        st.plan.close()


def test_allgather_from_host_buffers_edges():
    # a rank without host data sends its rows as they stand; a round without an output buffer
    w = W.small(W.C2, M=1024, N=2048, num_chunks=4)
    st = runner.make(w, fill_byte=5)
    S = w.slice_bytes
    try:
        host = [torch.from_numpy(H.fill_slice_bytes(w.dtype, w.seed, r, 1, w.M, w.N)).pin_memory()
                for r in range(w.P)]
        host[1] = None
        out = torch.zeros(w.buf_bytes, dtype=torch.uint8).pin_memory()
        assert st.plan.allgather_host(host, out, out_rank=0, stream=st.producer_stream).status == D.OK
        want = np.concatenate([h.numpy() if h is not None else np.full(S, 5, np.uint8) for h in host])
        np.testing.assert_array_equal(out.numpy(), want)
        host2 = [torch.from_numpy(H.fill_slice_bytes(w.dtype, w.seed, r, 2, w.M, w.N)).pin_memory()
                 for r in range(w.P)]
        assert st.plan.allgather_host(host2, None, stream=st.producer_stream).status == D.OK
        want2 = np.concatenate([h.numpy() for h in host2])
        for q in range(w.P):
            np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), want2)
    finally:
        st.plan.close()


# ---- plans sharing a copy stream ("Triggered Plans", The kernel author's contract: a plan
# whose copies wait behind an earlier plan's waiting copies cannot finish first) -------------
def _round1_everywhere(st, w):
    o = oracle_plan(w)
    assert oracle_round(o, w)[0] == OP.OK
    for q in range(w.P):
        np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"buffer {q}")


def test_close_behind_an_earlier_waiting_plan_leaves_it_closing():
    import time
    copy = torch.cuda.Stream()
    A = runner.make(WS, copy_stream=copy)
    B = runner.make(WS, copy_stream=copy, fill_byte=7)
    try:
        hA = A.plan.start(A.producer_stream)       # A's copier waits for A's producer
        hB = B.plan.start(B.producer_stream)       # B's copier is queued behind it
        D.dtt_fill_producer(B.buf_ptrs, B.desc, hB, B.producer_stream)
        t0 = time.perf_counter()
        assert B.plan.close() == D.RC_CLOSING      # returns at once, B cannot finish first
        assert time.perf_counter() - t0 < 1.0
        assert B.plan.state == D.CLOSING
        D.dtt_fill_producer(A.buf_ptrs, A.desc, hA, A.producer_stream)
        assert A.plan.close() == D.OK              # closing A finishes both
        assert B.plan.state == D.CLOSED
        _round1_everywhere(A, WS)
        _round1_everywhere(B, WS)
        assert B.plan.close() == D.OK              # releases B
        assert B.plan.state == D.CLOSED
    finally:
        A.plan.close()
        B.plan.close()


def test_closing_the_earlier_plan_does_not_wait_for_a_later_one():
    import time
    copy = torch.cuda.Stream()
    A = runner.make(WS, copy_stream=copy)
    B = runner.make(WS, copy_stream=copy)
    try:
        hA = A.plan.start(A.producer_stream)
        hB = B.plan.start(B.producer_stream)       # B's producer has not run yet
        D.dtt_fill_producer(A.buf_ptrs, A.desc, hA, A.producer_stream)
        t0 = time.perf_counter()
        assert A.plan.close() == D.OK              # drains A's copier only
        assert time.perf_counter() - t0 < 1.0
        D.dtt_fill_producer(B.buf_ptrs, B.desc, hB, B.producer_stream)
        rep = B.plan.wait()
        assert rep.status == D.OK and rep.copier_timeouts == 0
        _round1_everywhere(B, WS)
        B.plan.next_round()
        assert runner.run_round(B).status == D.OK  # B goes on alone
    finally:
        A.plan.close()
        B.plan.close()


def test_nested_plans_close_in_with_blocks():
    copy = torch.cuda.Stream()
    A = runner.make(WS, copy_stream=copy)
    B = runner.make(WS, copy_stream=copy)
    with A.plan:
        hA = A.plan.start(A.producer_stream)
        with B.plan:
            hB = B.plan.start(B.producer_stream)
            D.dtt_fill_producer(B.buf_ptrs, B.desc, hB, B.producer_stream)
        assert B.plan.state == D.CLOSING           # left the inner block behind A's copier
        D.dtt_fill_producer(A.buf_ptrs, A.desc, hA, A.producer_stream)
    assert B.plan.state == D.CLOSED                # the outer block's close finished it
    _round1_everywhere(B, WS)
    assert B.plan.close() == D.OK


def test_paced_producer_that_cannot_be_resident_is_rejected():
    # 8 ranks x 148 programs of 1024 threads cannot all be resident, so the pacing waits would
    # only run out: the launch is refused, and closing the plan still drains its copier
    w = W.Workload("pr", P=8, M=1024, N=1024, dtype=W.BF16, kind="tile_chunks", rounds=1, seed=31,
                   BM=128, BN=128, num_programs=148, tiles_per_chunk=148)
    st = runner.make(w, pace=2, threads=1024)
    try:
        h = st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        assert e.value.code == D.EINVAL
    finally:
        st.plan.close()


def test_prepare_all_gather_in_the_pages_form():
    # "Triggered Plans", section Model: schedules from each rank's own rows of its output (whole
    # by default, or chunks(mine, n, base=out)), the plan checking that they stay inside them; the
    # round's data (written here by the host, marked by dtt_publish) ends up everywhere
    P, M, N = 4, 64, 256
    outs = [torch.zeros(P * M, N, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    for scheds in (None, [D.chunks(outs[r][r * M:(r + 1) * M], 4, base=outs[r]) for r in range(P)]):
        plan = D.prepare_all_gather(outs, scheds)
        prod = torch.cuda.Stream()
        try:
            for R in (1, 2):
                h = plan.start(prod)
                with torch.cuda.stream(prod):
                    for r in range(P):
                        outs[r][r * M:(r + 1) * M] = float(10 * R + r)
                n_global = plan.info()[0]
                D.dtt_publish(h, 0, n_global, 0, prod)
                assert plan.wait().status == D.OK
                want = torch.cat([torch.full((M, N), float(10 * R + r), dtype=torch.bfloat16) for r in range(P)])
                for q in range(P):
                    assert torch.equal(outs[q].cpu(), want), (R, q)
                plan.next_round()
        finally:
            plan.close()
    # a schedule reaching into another rank's rows is refused at creation
    bad = [D.chunks(outs[r][0:2 * M], 2, base=outs[r]) for r in range(P)]
    with pytest.raises(D.DttError) as e:
        D.prepare_all_gather(outs, bad)
    assert e.value.code in (D.EOUTOFROWS, D.EOVERLAP)
