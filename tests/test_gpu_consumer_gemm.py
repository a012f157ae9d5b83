"""GPU: the consumer GEMM, the peer-kernel side of a triggered plan.  It is launched before the
producer, so it can only be right if every row block waits for its chunks: the producer's
values change every round, and a block read before its chunks arrived would hold the previous
round's data.  The product is checked against the oracle's fp64 product of the gathered buffer
the oracle computes for the same round (relative Frobenius error <= 1e-2)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import oracle_plan, oracle_round
from oracle import gemm as OG
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner

TOL = 1e-2


def _weights(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)


@pytest.mark.parametrize("q,N2,programs,bulk,M", [(0, 256, 0, None, 512), (3, 384, 7, None, 512),
                                                 (1, 128, 148, None, 512), (2, 256, 0, "full", 512),
                                                 (0, 256, 0, "small", 512), (3, 128, 0, "small", 512),
                                                 (1, 512, 2, None, 512), (2, 256, 7, None, 512),
                                                 (1, 256, 0, None, 160)])
def test_consumer_gemm_waits_for_its_rows(q, N2, programs, bulk, M):
    # bulk "full": the bulk-copy copier's 3 x 64 KiB ring leaves the GEMM no shared memory until
    # the copier's CTAs leave, so there is no overlap, but the result must be the same; "small":
    # a 2 x 32 KiB ring leaves room for the GEMM's shorter ring, and the two overlap.  N2 a
    # multiple of 256 over an even number of 128-row blocks runs the CTA-pair form (one pair with
    # 2 programs, three with 7); M = 160 gives 5 blocks, so the one-CTA form
    w = W.small(W.C2, M=M, N=1024, num_chunks=4 if M == 512 else 2, rounds=3)
    K = w.N
    rows = w.buf_bytes // (2 * K)
    Wt = _weights(N2, K, 77 + q)
    Wt_dev = Wt.cuda()
    out = torch.zeros(rows, N2, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    opts = {None: None,
            "full": D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=65536, stages=3),
            "small": D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=32768, stages=2)}[bulk]
    st = runner.make(w, opts=opts)                           # default: the vector copier
    o = oracle_plan(w)
    Wt64 = Wt.to(torch.float64).numpy()
    torch.cuda.synchronize()
    try:
        for R in (1, 2, 3):
            h = st.plan.start(st.producer_stream)
            if bulk != "full":
                st.plan.gemm_consumer(q, Wt_dev, out, N2, K, err, num_programs=programs, stream=cons)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            if bulk == "full":      # after the producer: nothing it needs queues behind the GEMM
                st.plan.gemm_consumer(q, Wt_dev, out, N2, K, err, num_programs=programs, stream=cons)
            rep = st.plan.wait()
            cons.synchronize()
            assert rep.status == D.OK and int(err.item()) == 0
            assert oracle_round(o, w)[0] == OP.OK
            X = torch.from_numpy(o.bufs[q].copy()).view(torch.bfloat16).view(rows, K)
            ref = OG.product(X.to(torch.float64).numpy(), Wt64)
            got = out.cpu().to(torch.float64).numpy()
            e = OG.rel_frobenius(got, ref)
            assert e <= TOL and e < 5e-3, (R, e)
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


def test_consumer_gemm_rejects_bad_shapes():
    w = W.small(W.C2, M=256, N=1024, num_chunks=2)
    st = runner.make(w)
    out = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wt = torch.zeros(128, 1024, dtype=torch.bfloat16, device="cuda")
    try:
        with pytest.raises(D.DttError) as e:            # not RUNNING
            st.plan.gemm_consumer(0, Wt, out, 128, 1024, err)
        assert e.value.code == D.ESTATE
        h = st.plan.start(st.producer_stream)
        with pytest.raises(D.DttError) as e:            # N not a multiple of 128
            st.plan.gemm_consumer(0, Wt, out, 100, 1024, err)
        assert e.value.code == D.EINVAL
        D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
        assert st.plan.wait().status == D.OK
    finally:
        st.plan.close()


def test_consumer_gemm_full_size_bench_launch():
    # The benchmark's consumer workload: rank 0's gathered c2 buffer X [16384, 4096] times
    # W^T [4096, 4096], the CTA-pair form launched right after plan_start, beside the vector
    # copier and the wave-ordered producer.  Every row is checked against the oracle's fp64
    # product of the same bf16 values (the gathered X from the C oracle's closed form).
    from oracle import cfill
    w = W.C2
    K, N2 = w.N, 4096
    rows = w.buf_bytes // (2 * K)
    launch = {k: v for k, v in runner.bench_launch(w, overlap=False).items() if k != "opts"}
    st = runner.make(w, opts=D.dtt_plan_opts_default(copier_threads=256), **launch)
    Wt = _weights(N2, K, 5)
    Wt_dev = Wt.cuda()
    Wt64 = Wt.to(torch.float64).numpy()
    out = torch.zeros(rows, N2, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        for R in (1, 2):
            h = st.plan.start(st.producer_stream)
            st.plan.gemm_consumer(0, Wt_dev, out, N2, K, err, stream=cons)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            rep = st.plan.wait()
            cons.synchronize()
            assert rep.status == D.OK and int(err.item()) == 0
            X = OG.bf16_bits_to_f64(cfill.expected_buffer(w, R).view(np.uint16).reshape(rows, K))
            ref = OG.product(X, Wt64)
            got = out.cpu().to(torch.float64).numpy()
            e = OG.rel_frobenius(got, ref)
            assert e <= TOL and e < 5e-3, (R, e)
            st.plan.next_round()
    finally:
        st.plan.close()


def _oracle_block_groups(o, block_bytes, nbytes):
    """The oracle's groups by position: block b holds every chunk with a byte in it (from the
    oracle's own chunk regions, row by row)."""
    nb = -(-nbytes // block_bytes)
    members = [[] for _ in range(nb)]
    for c, ch in enumerate(o.chunks):
        touched = set()
        for (off, rb, rows, pitch) in ch.regions:
            for i in range(rows):
                lo = off + i * pitch
                touched.update(range(lo // block_bytes, (lo + rb - 1) // block_bytes + 1))
        for b in touched:
            members[b].append(c)
    ids, groups = [], []
    for b in range(nb):
        if members[b]:
            ids.append(len(groups))
            groups.append(sorted(members[b]))
        else:
            ids.append(None)
    return groups, ids


GROUPED = {
    # chunks of exactly one 128-row block each; the pair form
    "chunks_pair": (W.small(W.C2, M=512, N=1024, num_chunks=4, rounds=3), 0, 256, 0),
    # 80-row chunks: blocks straddle two chunks and chunks two blocks; the one-CTA form
    "chunks_straddle": (W.small(W.C2, M=160, N=1024, num_chunks=2, rounds=3), 1, 256, 0),
    # tiles in the grouped order: a chunk's tiles lie in several blocks, a block's in several chunks
    "tiles_grouped": (W.Workload("tg", P=2, M=256, N=1024, dtype=W.BF16, kind="tile_chunks", rounds=3,
                                 seed=41, BM=64, BN=256, num_programs=3, tiles_per_chunk=3, group_m=2),
                      1, 384, 7),
}


@pytest.mark.parametrize("name", sorted(GROUPED))
def test_consumer_gemm_with_block_groups(name):
    # "Triggered Plans", Not supported yet, "Waiting on a group": one group per 128-row block of
    # X, so the GEMM waits once per block.  The groups equal the oracle's blocks-by-position, the
    # counters the oracle's after every round, and D the oracle's fp64 product
    w, q, N2, programs = GROUPED[name]
    K = w.N
    rows = w.buf_bytes // (2 * K)
    Wt = _weights(N2, K, 91)
    Wt_dev = Wt.cuda()
    out = torch.zeros(rows, N2, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cons = torch.cuda.Stream()
    st = runner.make(w)
    o = oracle_plan(w)
    groups, ids = _oracle_block_groups(o, 128 * 2 * K, w.buf_bytes)
    n, bg = st.plan.define_block_groups(128 * 2 * K)
    assert n == len(groups) and bg == ids
    o.define_groups(groups)
    Wt64 = Wt.to(torch.float64).numpy()
    torch.cuda.synchronize()
    try:
        for R in (1, 2, 3):
            h = st.plan.start(st.producer_stream)
            st.plan.gemm_consumer(q, Wt_dev, out, N2, K, err, num_programs=programs, stream=cons)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, st.producer_stream)
            rep = st.plan.wait()
            cons.synchronize()
            assert rep.status == D.OK and int(err.item()) == 0 and rep.device_status == 0
            assert oracle_round(o, w)[0] == OP.OK
            np.testing.assert_array_equal(st.plan.read_group_counters(), o.group_counters)
            X = torch.from_numpy(o.bufs[q].copy()).view(torch.bfloat16).view(rows, K)
            ref = OG.product(X.to(torch.float64).numpy(), Wt64)
            e = OG.rel_frobenius(out.cpu().to(torch.float64).numpy(), ref)
            assert e <= TOL and e < 5e-3, (R, e)
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()
