"""GPU: a user's own kernels drive a plan through the public device header alone
(`include/dtt_device.cuh`): a producer that writes its chunks and calls dtt_mark_ready, and a
consumer on a third stream, launched before the producer, that calls dtt_wait per chunk and
copies what arrived.  The kernels follow the header's contract for code that runs during a
round (loaded and given the library's shared-memory carveout before the first round).  They
are compiled here from tests/user_kernels.cu."""
import ctypes as C
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from conftest import ROOT

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D


def _build():
    out = os.path.join(tempfile.mkdtemp(prefix="dtt_user_"), "libuser.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "user_kernels.cu"), "-o", out], check=True)
    lib = C.CDLL(out)
    lib.user_kernels_prepare.restype = C.c_int
    lib.user_produce.argtypes = [C.POINTER(D.dtt_handle), C.c_void_p, C.c_uint64, C.c_void_p]
    lib.user_consume.argtypes = [C.POINTER(D.dtt_handle), C.c_void_p, C.c_void_p, C.c_uint64,
                                 C.c_uint64, C.c_void_p, C.c_void_p]
    lib.user_produce_paced.argtypes = [C.POINTER(D.dtt_handle), C.c_void_p, C.c_uint64, C.c_uint64,
                                       C.c_void_p, C.c_void_p, C.c_void_p]
    lib.user_probe.argtypes = [C.POINTER(D.dtt_handle), C.c_uint32, C.c_uint32, C.c_void_p,
                               C.c_void_p]
    lib.user_produce_reverse.argtypes = [C.POINTER(D.dtt_handle), C.c_void_p, C.c_uint64, C.c_uint64,
                                         C.c_void_p]
    lib.user_group_consume.argtypes = [C.POINTER(D.dtt_handle), C.c_uint32, C.c_void_p, C.c_void_p,
                                       C.c_uint64, C.c_void_p, C.c_void_p, C.c_uint64, C.c_void_p,
                                       C.c_void_p]
    lib.user_group_probe_launch.argtypes = [C.POINTER(D.dtt_handle), C.c_uint32, C.c_uint32, C.c_void_p,
                                            C.c_void_p]
    lib.user_probe_writable_launch.argtypes = [C.POINTER(D.dtt_handle), C.c_uint32, C.c_uint32, C.c_uint64,
                                               C.c_void_p, C.c_void_p, C.c_void_p]
    return lib


def _values(rank, rnd, n):
    """The bytes the user producer stores (the formula in user_kernels.cu, restated)."""
    i = np.arange(n, dtype=np.uint64)
    x = ((i * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    x ^= np.uint32((rank * 0x9E3779B9) & 0xFFFFFFFF) ^ np.uint32((rnd * 0x85EBCA6B) & 0xFFFFFFFF)
    x ^= x >> np.uint32(15)
    return (x & np.uint32(0xFF)).astype(np.uint8)


def test_user_producer_and_consumer_kernels():
    lib = _build()
    assert lib.user_kernels_prepare() == 0
    P, n, chunk = 3, 4, 1 << 20                  # 3 ranks x 4 chunks of 1 MiB
    S = n * chunk
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_chunks(r * S, n, chunk, chunk, n) for r in range(P)]
    plan = D.Plan(bufs, P * S, scheds, D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=65536,
                                                               stages=3))
    for s in scheds:
        s.free()
    q = 1                                        # the consuming rank
    dst = torch.zeros(P * S, dtype=torch.uint8, device="cuda")
    status = torch.full((P * n,), 99, dtype=torch.int32, device="cuda")
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        for rnd in (1, 2, 3):
            h = plan.start(prod)
            assert lib.user_consume(C.byref(h[q]), C.c_void_p(bufs[q].data_ptr()),
                                    C.c_void_p(dst.data_ptr()), chunk, 1 << 24,
                                    C.c_void_p(status.data_ptr()), C.c_void_p(cons.cuda_stream)) == 0
            for r in range(P):
                assert lib.user_produce(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S), chunk,
                                        C.c_void_p(prod.cuda_stream)) == 0
            rep = plan.wait()
            cons.synchronize()
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert status.cpu().tolist() == [0] * (P * n)
            want = np.concatenate([_values(r, rnd, S) for r in range(P)])
            np.testing.assert_array_equal(dst.cpu().numpy(), want)      # this round's data, all of it
            for b in bufs:
                np.testing.assert_array_equal(b.cpu().numpy(), want)
            plan.next_round()
    finally:
        plan.close()


def test_user_paced_producer_and_reusable():
    # Source side: dtt_reusable is false for every chunk before this round's marks, true for all
    # of them after wait(); a producer whose CTA c waits for chunk c - 1 to be reusable before it
    # writes chunk c finishes the round with this round's data everywhere, and each wait ended
    # only after chunk c - 1's arrival was signalled at every peer (gate timestamps).
    lib = _build()
    assert lib.user_kernels_prepare() == 0
    P, n, chunk = 3, 5, 1 << 20
    S = n * chunk
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_chunks(r * S, n, chunk, chunk, n) for r in range(P)]
    plan = D.Plan(bufs, P * S, scheds, D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=65536,
                                                               stages=3))
    for s in scheds:
        s.free()
    prod = torch.cuda.Stream()
    probe = torch.full((P, n), 7, dtype=torch.int32, device="cuda")
    wst = torch.full((P, n), 99, dtype=torch.int32, device="cuda")
    wend = torch.zeros((P, n), dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    try:
        for rnd in (1, 2, 3):
            h = plan.start(prod)
            for r in range(P):      # before any mark of this round
                assert lib.user_probe(C.byref(h[r]), h[r].first_chunk, n,
                                      C.c_void_p(probe[r].data_ptr()), C.c_void_p(prod.cuda_stream)) == 0
            for r in range(P):
                assert lib.user_produce_paced(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S),
                                              chunk, 1 << 24, C.c_void_p(wst[r].data_ptr()),
                                              C.c_void_p(wend[r].data_ptr()),
                                              C.c_void_p(prod.cuda_stream)) == 0
            rep = plan.wait()
            assert rep.status == D.OK and rep.device_status == 0
            prod.synchronize()
            assert probe.cpu().tolist() == [[0] * n] * P
            for r in range(P):
                assert lib.user_probe(C.byref(h[r]), h[r].first_chunk, n,
                                      C.c_void_p(probe[r].data_ptr()), C.c_void_p(prod.cuda_stream)) == 0
            prod.synchronize()
            assert probe.cpu().tolist() == [[1] * n] * P
            assert wst[:, 1:].cpu().tolist() == [[0] * (n - 1)] * P
            g = plan.read_gates()
            for r in range(P):
                for c in range(1, n):
                    prev = h[r].first_chunk + c - 1
                    arrivals = [int(g[q, prev, D.GATE_T_ARRIVE]) for q in range(P) if q != r]
                    assert int(wend[r, c]) >= max(arrivals) > 0, (rnd, r, c)
            want = np.concatenate([_values(r, rnd, S) for r in range(P)])
            for b in bufs:
                np.testing.assert_array_equal(b.cpu().numpy(), want)
            plan.next_round()
        # asking reusable of another rank's chunk is a misuse the round's wait reports
        h = plan.start(prod)
        assert lib.user_probe(C.byref(h[0]), h[1].first_chunk, 1, C.c_void_p(probe[0].data_ptr()),
                              C.c_void_p(prod.cuda_stream)) == 0
        for r in range(P):
            assert lib.user_produce_paced(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S), chunk,
                                          1 << 24, C.c_void_p(wst[r].data_ptr()),
                                          C.c_void_p(wend[r].data_ptr()), C.c_void_p(prod.cuda_stream)) == 0
        rep = plan.wait(raise_on_error=False)
        assert rep.status == D.EINVAL and rep.device_status & 1
        assert int(probe[0, 0].item()) == 0
    finally:
        plan.close()


@pytest.mark.parametrize("method", [1, 0, 2], ids=["bulk_copier", "vector_copier", "copy_engines"])
def test_out_of_order_producer_head_of_line(method):
    # "Triggered Plans", The kernel author's contract, item 1, and "Triggered SDMA Plans",
    # Testing (head-of-line ordering): a producer completes its chunks last to first.  The
    # result is still correct -- buffers and gate words 0-4 equal the oracle's for the same
    # order of marks -- only later: no chunk of a rank arrives anywhere before that rank's
    # first chunk (the head of its queues) has opened, although the others opened earlier.
    from oracle import plan as OP
    from oracle import schedule as OS
    lib = _build()
    assert lib.user_kernels_prepare() == 0
    P, n, chunk = 3, 4, 1 << 20
    S = n * chunk
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_chunks(r * S, n, chunk, chunk, n) for r in range(P)]
    opts = D.dtt_plan_opts_default(method=method, piece_bytes=65536, stages=3) if method == D.COPY_TMA \
        else D.dtt_plan_opts_default(method=method, copier_threads=256)
    opts.max_polls = 1 << 24         # the copy-engine proxy's bound: ~4 s
    plan = D.Plan(bufs, P * S, scheds, opts)
    for s_ in scheds:
        s_.free()
    # the oracle: same schedules, marks in the same (reverse) order, queues run after each mark
    o_bufs = [np.zeros(P * S, dtype=np.uint8) for _ in range(P)]
    o = OP.Plan(o_bufs, [OS.chunks(r * S, n, chunk, chunk, n) for r in range(P)])
    prod = torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        for rnd in (1, 2):
            h = plan.start(prod)
            for r in range(P):
                assert lib.user_produce_reverse(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S),
                                                chunk, 20000, C.c_void_p(prod.cuda_stream)) == 0
            rep = plan.wait()
            assert rep.status == D.OK and rep.copier_timeouts == 0
            o.start()
            log0 = len(o.delivery_log)
            for r in range(P):
                o.bufs[r][r * S:(r + 1) * S] = _values(r, rnd, S)
                for k in reversed(range(n)):
                    o.mark_ready(r, o.first[r] + k)
                    o.copier_progress()
                    if k > 0:           # head of line: nothing of rank r has moved yet
                        assert all(s != r for (s, _, _) in o.delivery_log[log0:])
            assert o.wait()[0] == OP.OK
            g = plan.read_gates()
            np.testing.assert_array_equal(g[:, :, :5], o.gates)
            for q in range(P):
                np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q])
            for r in range(P):
                head = h[r].first_chunk
                t_head = int(g[r, head, D.GATE_T_OPEN])
                opens = [int(g[r, head + k, D.GATE_T_OPEN]) for k in range(n)]
                assert opens == sorted(opens, reverse=True)      # they opened last to first
                assert opens[n - 1] + 3 * 20000 <= t_head         # ... with the spins between them
                for k in range(n):
                    for q in range(P):
                        if q != r:
                            assert int(g[q, head + k, D.GATE_T_ARRIVE]) >= t_head, (rnd, r, k, q)
            plan.next_round()
            o.next_round()
    finally:
        plan.close()


def test_group_waits_in_a_users_consumer_kernel():
    # "Triggered Plans", Not supported yet, "Waiting on a group": groups of chunks from several
    # source ranks (one of them the consumer's own), one wait each, in a consumer kernel launched
    # before the producers on a third stream.  Every group's data is this round's; the group
    # counters equal the oracle's (R * |g| at every rank); asking an undefined group is a misuse
    # that wait reports.
    from oracle import plan as OP
    from oracle import schedule as OS
    lib = _build()
    assert lib.user_kernels_prepare() == 0
    P, n, chunk = 3, 4, 1 << 18
    S = n * chunk
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_chunks(r * S, n, chunk, chunk, n) for r in range(P)]
    plan = D.Plan(bufs, P * S, scheds, D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=65536, stages=3))
    for s_ in scheds:
        s_.free()
    groups = [[0, 4, 8], [1, 2, 3], list(range(P * n)), [7], [11, 5, 9, 1]]
    assert plan.define_groups(groups) == len(groups)
    with pytest.raises(D.DttError) as e:
        plan.define_groups(groups)                       # once per plan
    assert e.value.code == D.ESTATE
    o = OP.Plan([np.zeros(P * S, dtype=np.uint8) for _ in range(P)],
                [OS.chunks(r * S, n, chunk, chunk, n) for r in range(P)])
    o.define_groups(groups)
    goff = torch.tensor(np.cumsum([0] + [len(g) for g in groups]), dtype=torch.int32, device="cuda")
    gids = torch.tensor([c for g in groups for c in g], dtype=torch.int32, device="cuda")
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    dst = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    status = torch.full((P, len(groups)), 99, dtype=torch.int32, device="cuda")
    probe = torch.full((len(groups),), 7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    try:
        for rnd in (1, 2, 3):
            h = plan.start(prod)
            assert lib.user_group_probe_launch(C.byref(h[0]), 0, len(groups), C.c_void_p(probe.data_ptr()),
                                               C.c_void_p(prod.cuda_stream)) == 0
            for q in range(P):
                assert lib.user_group_consume(C.byref(h[q]), len(groups), C.c_void_p(bufs[q].data_ptr()),
                                              C.c_void_p(dst[q].data_ptr()), chunk, C.c_void_p(goff.data_ptr()),
                                              C.c_void_p(gids.data_ptr()), 1 << 24,
                                              C.c_void_p(status[q].data_ptr()), C.c_void_p(cons.cuda_stream)) == 0
            for r in range(P):
                assert lib.user_produce(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S), chunk,
                                        C.c_void_p(prod.cuda_stream)) == 0
            rep = plan.wait()
            cons.synchronize()
            assert rep.status == D.OK and rep.device_status == 0
            assert probe.cpu().tolist() == [0] * len(groups)      # before this round's marks
            assert status.cpu().tolist() == [[0] * len(groups)] * P
            want = np.concatenate([_values(r, rnd, S) for r in range(P)])
            for q in range(P):
                got = dst[q].cpu().numpy()
                for g in groups:
                    for c in g:
                        np.testing.assert_array_equal(got[c * chunk:(c + 1) * chunk], want[c * chunk:(c + 1) * chunk])
            o.start()
            for r in range(P):
                o.bufs[r][r * S:(r + 1) * S] = _values(r, rnd, S)
                for c in o.chunks_of(r):
                    o.mark_ready(r, c)
            o.copier_progress()
            assert o.wait()[0] == OP.OK
            np.testing.assert_array_equal(plan.read_group_counters(), o.group_counters)
            np.testing.assert_array_equal(plan.read_gates()[:, :, :5], o.gates)
            plan.next_round()
            o.next_round()
        # a group the plan does not have: the wait gives up at once and wait() reports the misuse
        h = plan.start(prod)
        assert lib.user_group_probe_launch(C.byref(h[1]), len(groups), 1, C.c_void_p(probe.data_ptr()),
                                           C.c_void_p(prod.cuda_stream)) == 0
        for r in range(P):
            assert lib.user_produce(C.byref(h[r]), C.c_void_p(bufs[r].data_ptr() + r * S), chunk,
                                    C.c_void_p(prod.cuda_stream)) == 0
        rep = plan.wait(raise_on_error=False)
        assert rep.status == D.EINVAL and rep.device_status & 2
        assert int(probe[0].item()) == 0
    finally:
        plan.close()


def test_writable_with_overlapping_rounds():
    # Overlapping rounds (opts.overlap): round 1 marks every chunk but rank 0's second one, so
    # its copier delivers rank 0's first chunk and gives that one up.  With round 2 started
    # behind it, rank 0's first chunk is writable (its round-1 copies landed) and the second is
    # not: a bounded dtt_wait_writable on it returns DTT_ETIMEDOUT.  Round 1's check names the
    # unmarked chunk, as the oracle's overlapped plan does.
    from oracle import plan as OP
    from oracle import schedule as OS
    lib = _build()
    assert lib.user_kernels_prepare() == 0
    P, n, chunk = 2, 2, 1 << 16
    S = n * chunk
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scheds = [D.dtt_schedule_chunks(r * S, n, chunk, chunk, n) for r in range(P)]
    plan = D.Plan(bufs, P * S, scheds, D.dtt_plan_opts_default(overlap=1, max_polls=1 << 12))
    for s in scheds:
        s.free()
    o = OP.Plan([np.zeros(1, dtype=np.uint8) for _ in range(P)],
                [OS.chunks(r * S, n, chunk, chunk, n) for r in range(P)], validate=False, copy_data=False,
                overlap=True)
    prod = torch.cuda.Stream()
    now = torch.full((n,), 7, dtype=torch.int32, device="cuda")
    waited = torch.full((n,), 7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    try:
        h = plan.start(prod)
        o.start()
        for c in (0, 2, 3):                   # chunk 1 (rank 0's second) is never marked
            D.dtt_publish(h, c, 1, 0, prod)
            o.mark_ready(o.owner[c], c)
        plan.next_round()
        o.next_round()
        h = plan.start(prod)
        o.start()
        o.copier_progress()
        torch.cuda.synchronize()              # round 1's copier has delivered or given up
        assert lib.user_probe_writable_launch(C.byref(h[0]), h[0].first_chunk, n, 4096,
                                              C.c_void_p(now.data_ptr()), C.c_void_p(waited.data_ptr()),
                                              C.c_void_p(prod.cuda_stream)) == 0
        prod.synchronize()
        assert now.cpu().tolist() == [int(o.writable(0, 0, 2)), int(o.writable(0, 1, 2))] == [1, 0]
        assert waited.cpu().tolist() == [0, D.ETIMEDOUT]
        assert o.wait() == (OP.TIMEOUT, [1], [])
        rep = plan.wait(raise_on_error=False)
        assert rep.status == D.ETIMEDOUT and rep.round == 1 and rep.shorts == [1]
    finally:
        plan.close()
