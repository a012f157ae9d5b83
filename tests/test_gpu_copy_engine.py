"""GPU: the copy-engine transport (opts.method = DTT_COPY_ENGINE) against the oracle.

The pages' copy engine runs POLL_REGMEM (ready >= round) -> COPY -> ATOMIC (arrival += 1) chains
("Triggered Plans", introduction).  Here a host proxy thread polls mapped gate words, issues the
copies on the GPU's copy engines, one stream per (source, peer) queue, and a one-warp kernel adds
each chunk's arrivals.  Results must be those of the SM copiers: every buffer byte and gate word
equal to the oracle's, head-of-line order per queue, timeouts naming the short chunks.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import assert_buffers_equal, expected_on_device, oracle_plan, oracle_round
from oracle import hashfill as H
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner


def _ce(**kw):
    return D.dtt_plan_opts_default(method=D.COPY_ENGINE, **kw)


def _parity(w, rounds, **launch):
    st = runner.make(w, opts=_ce(), **launch)
    o = oracle_plan(w)
    try:
        for R in range(1, rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w) == (OP.OK, [], [])
            for q in range(w.P):
                np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"round {R} buffer {q}")
            g = st.plan.read_gates()
            np.testing.assert_array_equal(g[:, :, :5], o.gates)
            for c in range(o.G):            # every arrival stamped after its gate opened
                s = o.owner[c]
                for p in range(w.P):
                    if p != s:
                        assert int(g[p, c, D.GATE_T_ARRIVE]) >= int(g[s, c, D.GATE_T_OPEN]) > 0
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


SMALL = {
    "chunks_ragged": (W.small(W.C2, M=70, N=256, num_chunks=8), {}),
    "tiles_grouped_ragged": (W.Workload("t", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks", rounds=3,
                                        seed=7, BM=64, BN=48, num_programs=5, tiles_per_chunk=5, group_m=2), {}),
    "tiles_unaligned": (W.Workload("u", P=2, M=37, N=203, dtype=W.BF16, kind="tile_chunks", rounds=2, seed=8,
                                   BM=16, BN=40, num_programs=3, tiles_per_chunk=4), {}),
    "whole_f32_8writers": (W.small(W.C4A, M=64, N=64, rounds=3), {}),
    "bcast_u8": (W.Workload("b", P=4, M=64, N=4096, dtype=W.U8, kind="whole", rounds=2, seed=9,
                            num_programs=8, broadcast=True), {}),
    "chunks_group5": (W.small(W.C2, M=256, N=512, num_chunks=4), {"group": 5, "programs": 1}),
    "single_rank": (W.Workload("s1", P=1, M=64, N=256, dtype=W.BF16, kind="chunks", rounds=2, seed=21,
                               num_chunks=4), {}),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_copy_engine_parity_small(name):
    w, kw = SMALL[name]
    _parity(w, min(w.rounds, 3), **kw)


def test_copy_engine_c2_full_size():
    # the benchmark's c2 producer (chunks opening wave by wave) with the copy engines moving them:
    # every byte of every buffer against the oracle's closed form, and the gates
    w = W.C2
    launch = {k: v for k, v in runner.bench_launch(w, overlap=False).items() if k != "opts"}
    st = runner.make(w, opts=_ce(), **launch)
    o = oracle_plan(w, copy_data=False)
    try:
        for R in range(1, 4):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w)[0] == OP.OK
            assert_buffers_equal(st.bufs, expected_on_device(w, R), f"round {R}")
            np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


WS = W.Workload("p", P=2, M=64, N=128, dtype=W.BF16, kind="chunks", rounds=3, seed=21, num_chunks=2)


def test_copy_engine_missing_mark_times_out_head_of_line():
    # rank 1's first chunk is never marked: its second chunk, though ready, waits behind it on
    # the queue (head of line), and wait() names both, as the oracle does
    st = runner.make(WS, opts=_ce(max_polls=20000))
    o = oracle_plan(WS)
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_publish(h, 0, 2, 0, st.producer_stream)
        D.dtt_publish(h, 3, 1, 0, st.producer_stream)
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
        np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
    finally:
        st.plan.close()


def test_copy_engine_extra_mark_is_reported():
    st = runner.make(WS, opts=_ce())
    try:
        h = st.plan.start(st.producer_stream)
        D.dtt_fill_producer(st.bufs, st.desc, h, st.producer_stream)
        D.dtt_publish(h, 1, 1, 1, st.producer_stream)
        rep = st.plan.wait(raise_on_error=False)
        assert rep.status == D.EEXTRA and rep.extras == [1]
    finally:
        st.plan.close()


def test_copy_engine_close_mid_round_sends_chunks_as_they_stand():
    st = runner.make(WS, opts=_ce())
    o = oracle_plan(WS)
    data = torch.arange(WS.slice_bytes, dtype=torch.int64).remainder(251).to(torch.uint8).cuda()
    st.producer_stream.wait_stream(torch.cuda.current_stream())
    h = st.plan.start(st.producer_stream)
    with torch.cuda.stream(st.producer_stream):
        st.bufs[0][:WS.slice_bytes // 2].copy_(data[:WS.slice_bytes // 2])
    D.dtt_publish(h, 0, 1, 0, st.producer_stream)
    st.plan.close()
    torch.cuda.synchronize()
    o.start()
    o.bufs[0][:WS.slice_bytes // 2] = data[:WS.slice_bytes // 2].cpu().numpy()
    o.mark_ready(0, 0)
    o.close()
    for q in range(2):
        np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q])


def test_copy_engine_group_counters_and_consumer_gather():
    # groups with the copy-engine transport: the signal kernel counts arrivals in the peers'
    # group counters as the SM copier does; a consumer kernel's per-chunk waits read this round's
    # data
    w = W.small(W.C2, M=96, N=512, num_chunks=3)
    st = runner.make(w, opts=_ce())
    o = oracle_plan(w)
    groups = [[0, 4, 8], [1, 2, 3, 11], list(range(12)), [5]]
    st.plan.define_groups(groups)
    o.define_groups(groups)
    dst = torch.zeros(w.buf_bytes, dtype=torch.uint8, device="cuda")
    status = torch.full((12,), 99, dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        for R in (1, 2):
            h = st.plan.start(st.producer_stream)
            st.plan.consumer_gather(2, dst, 1 << 24, status, 8, cons)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            rep = st.plan.wait()
            cons.synchronize()
            assert rep.status == D.OK
            assert oracle_round(o, w)[0] == OP.OK
            np.testing.assert_array_equal(st.plan.read_group_counters(), o.group_counters)
            assert status.cpu().tolist() == [0] * 12
            got, want = dst.cpu().numpy(), o.bufs[2]
            S = w.slice_bytes
            for r in range(w.P):
                if r != 2:
                    np.testing.assert_array_equal(got[r * S:(r + 1) * S], want[r * S:(r + 1) * S])
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


def test_copy_engine_rejects_host_buffer_rounds():
    st = runner.make(WS, opts=_ce())
    try:
        with pytest.raises(D.DttError) as e:
            st.plan.allgather_host([None, None], None, 0, st.producer_stream)
        assert e.value.code == D.EINVAL
    finally:
        st.plan.close()
