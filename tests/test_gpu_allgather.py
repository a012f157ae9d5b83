"""GPU parity: the CUDA triggered all-gather (copier, fill producer, gates, check) against the
CPU oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import assert_buffers_equal, expected_on_device, oracle_plan, oracle_round
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner


def _gates_match(st, o):
    g = st.plan.read_gates()
    assert g.shape[:2] == o.gates.shape[:2]
    np.testing.assert_array_equal(g[:, :, :5], o.gates)
    return g


def run_parity(w, rounds, opts=None, cluster=1, programs=None, threads=0, group=1, pace=0):
    st = runner.make(w, opts=opts, cluster=cluster, programs=programs, threads=threads, group=group,
                     pace=pace)
    o = oracle_plan(w)
    try:
        for R in range(1, rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w) == (OP.OK, [], [])
            for q in range(w.P):
                np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q],
                                              err_msg=f"round {R} buffer {q}")
            g = _gates_match(st, o)
            t_open, t_arr = g[:, :, D.GATE_T_OPEN], g[:, :, D.GATE_T_ARRIVE]
            for c in range(o.G):
                s = o.owner[c]
                for p in range(w.P):
                    if p != s:
                        assert int(t_arr[p, c]) >= int(t_open[s, c]) > 0
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


SMALL = {
    "c1": (W.C1, {}),
    "chunks_ragged": (W.small(W.C2, M=70, N=256, num_chunks=8), {}),
    "tiles_grouped_ragged": (W.Workload("t", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                        rounds=3, seed=7, BM=64, BN=48, num_programs=5,
                                        tiles_per_chunk=5, group_m=2), {}),
    "tiles_unaligned": (W.Workload("u", P=2, M=37, N=203, dtype=W.BF16, kind="tile_chunks",
                                   rounds=2, seed=8, BM=16, BN=40, num_programs=3,
                                   tiles_per_chunk=4), {}),
    "whole_f32_8writers": (W.small(W.C4A, M=64, N=64, rounds=4), {}),
    "bcast_u8": (W.Workload("b", P=4, M=64, N=4096, dtype=W.U8, kind="whole", rounds=2, seed=9,
                            num_programs=8, broadcast=True), {}),
    "chunks_cluster4": (W.small(W.C2, M=256, N=512, num_chunks=4), {"cluster": 4}),
    "tiles_cluster2": (W.Workload("t2", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                  rounds=2, seed=10, BM=64, BN=48, num_programs=5,
                                  tiles_per_chunk=5, group_m=2), {"cluster": 2}),
    "small_pieces_few_ctas": (W.small(W.C2, M=64, N=1024, num_chunks=4),
                              {"opts": dict(piece_bytes=4096, copier_ctas=7, copier_threads=128)}),
    "many_ctas": (W.small(W.C2, M=32, N=256, num_chunks=2),
                  {"opts": dict(copier_ctas=600, copier_threads=64)}),
    # the bulk-copy (TMA) copier: 1D pieces, per-row 2D pieces, a broadcast, few stages
    "bulk_chunks_ragged": (W.small(W.C2, M=70, N=256, num_chunks=8),
                           {"opts": dict(method=1, piece_bytes=16384)}),
    "bulk_tiles_grouped": (W.Workload("tb", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                      rounds=3, seed=11, BM=64, BN=48, num_programs=5,
                                      tiles_per_chunk=5, group_m=2),
                           {"opts": dict(method=1, piece_bytes=8192, stages=4)}),
    # 2D windows as tensor-map boxes: boxes taller than 256 rows are split, rows over 2 KiB
    # go row by row, clipped edge tiles get boxes of their own shape
    "bulk_tall_tiles": (W.Workload("tt", P=2, M=700, N=64, dtype=W.BF16, kind="tile_chunks",
                                   rounds=2, seed=14, BM=320, BN=16, num_programs=4,
                                   tiles_per_chunk=4), {"opts": dict(method=1)}),
    "bulk_wide_tiles": (W.Workload("tw", P=3, M=40, N=2400, dtype=W.BF16, kind="tile_chunks",
                                   rounds=2, seed=15, BM=16, BN=1104, num_programs=3,
                                   tiles_per_chunk=2), {"opts": dict(method=1, piece_bytes=65536)}),
    "bulk_whole_f32": (W.small(W.C4A, M=64, N=64, rounds=3),
                       {"opts": dict(method=1, piece_bytes=4096, stages=2, copier_ctas=5)}),
    "bulk_bcast_u8": (W.Workload("bb", P=4, M=64, N=4096, dtype=W.U8, kind="whole", rounds=2,
                                 seed=12, num_programs=8, broadcast=True),
                      {"opts": dict(method=1, piece_bytes=32768, stages=6)}),
    # group writers: several CTAs anywhere on the GPU write a step and mark it once
    "chunks_group5": (W.small(W.C2, M=256, N=512, num_chunks=4), {"group": 5, "programs": 1}),
    "chunks_group3_bulk": (W.small(W.C2, M=96, N=1024, num_chunks=6),
                           {"group": 3, "programs": 2,
                            "opts": dict(method=1, piece_bytes=16384, stages=4)}),
    "tiles_group3": (W.Workload("tg", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                rounds=3, seed=13, BM=64, BN=48, num_programs=5,
                                tiles_per_chunk=5, group_m=2), {"group": 3}),
    "whole_f32_8writers_group4": (W.small(W.C4A, M=64, N=64, rounds=3),
                                  {"group": 4, "opts": dict(method=1, piece_bytes=4096, stages=4)}),
    "whole_1writer_group16": (W.small(W.C1, M=200), {"group": 16, "threads": 512}),
    # one rank: no peers, so nothing is copied, but every chunk must still be marked, opened
    # and counted complete (completion stays 0: P - 1 = 0 deliveries)
    "single_rank_vec": (W.Workload("s1", P=1, M=64, N=256, dtype=W.BF16, kind="chunks", rounds=3,
                                   seed=21, num_chunks=4), {}),
    "single_rank_bulk": (W.Workload("s1b", P=1, M=64, N=256, dtype=W.BF16, kind="tile_chunks",
                                    rounds=3, seed=22, BM=16, BN=64, num_programs=3,
                                    tiles_per_chunk=3), {"opts": dict(method=1, piece_bytes=4096)}),
    # a paced producer: a program writes chunk k once chunk k - pace of its rank is delivered
    "tiles_paced2_bulk": (W.Workload("tp", P=4, M=512, N=512, dtype=W.BF16, kind="tile_chunks",
                                     rounds=3, seed=16, BM=64, BN=64, num_programs=6,
                                     tiles_per_chunk=6, group_m=3),
                          {"pace": 2, "threads": 128,
                           "opts": dict(method=1, piece_bytes=8192, stages=2, ctas_per_sm=3)}),
    "chunks_paced1": (W.small(W.C2, M=96, N=1024, num_chunks=6), {"pace": 1, "programs": 2}),
    "tiles_paced1_group3": (W.Workload("tq", P=3, M=300, N=200, dtype=W.BF16, kind="tile_chunks",
                                       rounds=3, seed=17, BM=64, BN=48, num_programs=5,
                                       tiles_per_chunk=5, group_m=2), {"group": 3, "pace": 1}),
    # pacing with the copier started after the producer: every pacing wait runs out (about a
    # millisecond each) and the producer goes on; the data and gates are the same
    "paced_copier_after_producer": (W.small(W.C2, M=64, N=512, num_chunks=4),
                                    {"pace": 1, "programs": 1,
                                     "opts": dict(deferred_copier=1)}),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_small(name):
    w, kw = SMALL[name]
    kw = dict(kw)
    opts = kw.pop("opts", None)
    run_parity(w, min(w.rounds, 3), opts=D.dtt_plan_opts_default(**opts) if opts else None, **kw)


def test_parity_c1_full():
    run_parity(W.C1, W.C1.rounds)


def test_parity_c1_full_bench_launch():
    run_parity(W.C1, W.C1.rounds, **runner.bench_launch(W.C1))


def test_parity_c4a_full_stale_data_check():
    # 8 writers on one 4 MiB gate per rank, values change every round: a stale copy fails
    run_parity(W.C4A, W.C4A.rounds)


def test_parity_c4a_full_bench_launch():
    # the benchmark's launch: each of the 8 writers is a group of CTAs marking once
    run_parity(W.C4A, 4, **runner.bench_launch(W.C4A))


def _run_full(w, rounds, launch):
    """The workload at full size, every byte of every buffer against the oracle every round."""
    st = runner.make(w, **launch)
    o = oracle_plan(w, copy_data=False)
    try:
        for R in range(1, rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w)[0] == OP.OK
            assert_buffers_equal(st.bufs, expected_on_device(w, R), f"{w.name} round {R}")
            _gates_match(st, o)
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


def test_parity_c2_full_bench_launch():
    _run_full(W.C2, W.C2.rounds, runner.bench_launch(W.C2))


def test_parity_c3_full():
    _run_full(W.C3, W.C3.rounds, runner.bench_launch(W.C3))


def test_parity_c4b_broadcast_full():
    w = W.C4B
    st = runner.make(w, **runner.bench_launch(w))
    o = oracle_plan(w, copy_data=False)
    try:
        assert st.plan.info()[0] == 1
        rep = runner.run_round(st)
        assert rep.status == D.OK and rep.copier_timeouts == 0
        assert oracle_round(o, w)[0] == OP.OK
        assert_buffers_equal(st.bufs, expected_on_device(w, 1), w.name)
        _gates_match(st, o)
    finally:
        st.plan.close()


def test_broadcast_split_into_1gib_copies():
    s = runner.schedules_for(W.C4B)
    regs, writers = s[0].chunk(0)
    assert [r[1] for r in regs] == [1 << 30, 1 << 30, 1 << 29]
    assert all(x.n_chunks == 0 for x in s[1:])


def test_parity_c2_full_bulk_copier():
    launch = dict(runner.bench_launch(W.C2))
    launch["opts"] = D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=16384, stages=8)
    _run_full(W.C2, 3, launch)


def test_parity_c3_full_vector_copier():
    # the bench launch moves c3's tiles as tensor-map boxes; this is the 16-byte vector path
    launch = dict(runner.bench_launch(W.C3))
    launch["opts"] = D.dtt_plan_opts_default(method=D.COPY_VEC16, copier_threads=256)
    _run_full(W.C3, 3, launch)


def test_bulk_copier_rejects_unaligned_regions():
    w = SMALL["tiles_unaligned"][0]
    with pytest.raises(D.DttError) as e:
        runner.make(w, opts=D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=16384))
    assert e.value.code == D.EINVAL


def test_many_rounds_keep_the_gates_and_data_right():
    # 500 rounds of the benchmark's launch back to back: the gates follow the closed form of the
    # round count, and the data is the last round's everywhere (every byte)
    w = W.C2
    R = 500
    st = runner.make(w, **runner.bench_launch(w))
    try:
        for r in range(1, R + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0, r
            if r < R:
                st.plan.next_round()
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


def test_pacing_stalls_at_most_once_per_program():
    # A paced producer whose copier runs only after it (deferred_copier = 1): every pacing wait
    # would run out.  A program stops pacing after its first wait runs out, so a round with 8
    # chunks per rank costs about one stall (~1 ms), not seven; the data is the oracle's.
    import time

    def round_ms(w, pace):
        st = runner.make(w, pace=pace, programs=1, opts=D.dtt_plan_opts_default(deferred_copier=1))
        o = oracle_plan(w)
        try:
            times = []
            for R in range(1, 4):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                rep = runner.run_round(st)
                times.append((time.perf_counter() - t0) * 1e3)
                assert rep.status == D.OK
                assert oracle_round(o, w)[0] == OP.OK
                for q in range(w.P):
                    np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q])
                st.plan.next_round()
                o.next_round()
            return min(times)
        finally:
            st.plan.close()

    w8 = W.small(W.C2, M=64, N=512, num_chunks=8)
    w2 = W.small(W.C2, M=64, N=512, num_chunks=2)
    stall8 = round_ms(w8, 1) - round_ms(w8, 0)
    stall2 = round_ms(w2, 1) - round_ms(w2, 0)
    print(f"pacing stall per round: 8 chunks {stall8:.2f} ms, 2 chunks {stall2:.2f} ms")
    assert stall2 > 0.2                      # the one stall is there ...
    assert stall8 < 2.0 * stall2 + 0.5       # ... and 7 waits did not become 7 stalls
