"""GPU: other destinations ("Triggered Plans", Not supported yet: a copy landing at another
offset, pitch or buffer, and a chunk going to only some peers -- what reduce-scatter needs)
against the oracle, on the vector, bulk-copy and copy-engine transports: every byte of every
buffer (and destination buffer) and the gate words 0-4."""
import numpy as np
import pytest
import torch

from oracle import hashfill as H
from oracle import plan as OP
from oracle import schedule as OS

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D

TRANSPORTS = {"vector": dict(method=0, copier_threads=256),
              "bulk": dict(method=1, piece_bytes=16384, stages=2),
              "copy_engines": dict(method=2)}


def _opts(transport, **kw):
    o = dict(TRANSPORTS[transport])
    o.update(kw)
    return D.dtt_plan_opts_default(allgather=0, **o)


class Case:
    """P ranks, each filling rows [0, M) of N bf16 at the start of its buffer with the oracle's
    hashed values (the library's fill producer), in blocks of `rows` rows; `chunk_of(s, b)` gives
    block b of rank s as (dests or None, peers).  buf_bytes per buffer; dst_bytes > 0: separate
    destination buffers."""

    def __init__(self, P, M, N, rows, buf_bytes, chunk_of, dst_bytes=0, seed=77):
        self.P, self.M, self.N, self.rows = P, M, N, rows
        self.rb = N * 2
        self.buf_bytes, self.dst_bytes, self.seed = buf_bytes, dst_bytes, seed
        self.nblocks = M // rows
        self.spec = [[chunk_of(s, b) for b in range(self.nblocks)] for s in range(P)]

    def region(self, b):
        return (b * self.rows * self.rb, self.rows * self.rb, 1, self.rows * self.rb)

    def oracle(self, overlap=False):
        scheds = [OS.Schedule([OS.Chunk([self.region(b)], 1, dests=d, peers=(m or None))
                               for b, (d, m) in enumerate(self.spec[s])]) for s in range(self.P)]
        bufs = [np.zeros(self.buf_bytes, dtype=np.uint8) for _ in range(self.P)]
        dst = [np.zeros(self.dst_bytes, dtype=np.uint8) for _ in range(self.P)] if self.dst_bytes else None
        return OP.Plan(bufs, scheds, allgather=False, dst_bufs=dst, overlap=overlap)

    def library(self, transport, overlap=False):
        scheds = []
        for s in range(self.P):
            sc = D.dtt_schedule_empty()
            for b, (d, m) in enumerate(self.spec[s]):
                sc.add_chunk([self.region(b)], 1, dests=d, peers=m)
            scheds.append(sc)
        bufs = [torch.zeros(self.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(self.P)]
        dst = [torch.zeros(self.dst_bytes, dtype=torch.uint8, device="cuda") for _ in range(self.P)] \
            if self.dst_bytes else None
        plan = D.Plan(bufs, self.buf_bytes, scheds, _opts(transport, overlap=int(overlap)), dst_bufs=dst,
                      dst_bytes=self.dst_bytes)
        for sc in scheds:
            sc.free()
        desc = D.fill_desc("bf16", self.seed, self.M, self.N, self.rb, self.buf_bytes, [0] * self.P,
                           self.rows, self.N, 1, 1, mark_mode=D.MARK_PER_STEP)
        torch.cuda.synchronize()
        return plan, bufs, dst, desc

    def run(self, transport, rounds=3, groups=None):
        plan, bufs, dst, desc = self.library(transport)
        o = self.oracle()
        if groups is not None:
            plan.define_groups(groups)
            o.define_groups(groups)
        prod = torch.cuda.Stream()
        try:
            for R in range(1, rounds + 1):
                h = plan.start(prod)
                D.dtt_fill_producer(bufs, desc, h, prod)
                rep = plan.wait()
                assert rep.status == D.OK and rep.copier_timeouts == 0
                o.start()
                for s in range(self.P):
                    o.bufs[s][:self.M * self.rb] = H.fill_slice_bytes("bf16", self.seed, s, R, self.M, self.N)
                    for c in o.chunks_of(s):
                        o.mark_ready(s, c)
                o.copier_progress()
                assert o.wait()[0] == OP.OK
                for q in range(self.P):
                    np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"{transport} R{R} buf {q}")
                    if dst:
                        np.testing.assert_array_equal(dst[q].cpu().numpy(), o.dst[q], err_msg=f"{transport} R{R} dst {q}")
                np.testing.assert_array_equal(plan.read_gates()[:, :, :5], o.gates)
                if groups is not None:
                    np.testing.assert_array_equal(plan.read_group_counters(), o.group_counters)
                plan.next_round()
                o.next_round()
        finally:
            plan.close()


    def run_overlapped(self, transport, rounds=4):
        """Rounds two at a time (opts.overlap) on the library and the oracle through the same
        host calls; every buffer, destination buffer and gate word after the last round."""
        plan, bufs, dst, desc = self.library(transport, overlap=True)
        o = self.oracle(overlap=True)
        prod = torch.cuda.Stream()
        try:
            for i in range(rounds):
                R = i + 1
                h = plan.start(prod)
                D.dtt_fill_producer(bufs, desc, h, prod)
                assert o.start() == R
                for s in range(self.P):
                    data = np.zeros(self.buf_bytes, dtype=np.uint8)
                    data[:self.M * self.rb] = H.fill_slice_bytes("bf16", self.seed, s, R, self.M, self.N)
                    for c in o.chunks_of(s):
                        while not o.writable(s, c, R):
                            assert o.copier_progress() > 0
                        o.write_chunk(s, c, data, R)
                        o.mark_ready(s, c, R)
                if plan.pending:
                    rep = plan.wait()
                    assert rep.status == D.OK and rep.round == R - 1 and rep.copier_timeouts == 0
                    o.copier_progress()
                    assert o.wait()[0] == OP.OK
                if i + 1 < rounds:
                    plan.next_round()
                    o.next_round()
            rep = plan.wait()
            assert rep.status == D.OK and rep.round == rounds
            o.copier_progress()
            assert o.wait()[0] == OP.OK
            for q in range(self.P):
                np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"{transport} buf {q}")
                if dst:
                    np.testing.assert_array_equal(dst[q].cpu().numpy(), o.dst[q], err_msg=f"{transport} dst {q}")
            np.testing.assert_array_equal(plan.read_gates()[:, :, :5], o.gates)
        finally:
            plan.close()


def _reduce_scatter(P=4, rows=64, N=256, separate=False):
    """Block b of every rank goes only to rank b, into rank b's staging slot of the sender (after
    the partials in place, or at the start of a separate destination buffer)."""
    rb = N * 2
    B = rows * rb
    M = P * rows
    base = 0 if separate else P * B

    def chunk_of(s, b):
        return [(base + s * B, B)], (1 << b)      # b == s: only the owner's bit, so nobody
    return Case(P, M, N, rows, 2 * P * B, chunk_of, dst_bytes=P * B if separate else 0)


@pytest.mark.parametrize("transport", sorted(TRANSPORTS))
@pytest.mark.parametrize("separate", [False, True], ids=["in_place", "staging_buffers"])
def test_reduce_scatter_into_staging_slots(transport, separate):
    _reduce_scatter(separate=separate).run(transport)


@pytest.mark.parametrize("transport", sorted(TRANSPORTS))
@pytest.mark.parametrize("separate", [False, True], ids=["in_place", "staging_buffers"])
def test_reduce_scatter_overlapped_rounds(transport, separate):
    # overlapping rounds: a round's partial blocks are written while the previous round's are
    # still being sent to their owners' slots
    _reduce_scatter(separate=separate).run_overlapped(transport)


@pytest.mark.parametrize("transport", sorted(TRANSPORTS))
def test_gather_to_pitched_destination(transport):
    # every block goes to every other rank, landing as a 2D window of its rows with a wider pitch
    # in a separate buffer: rank s's block b at rows [(s*nb + b)*rows...) of a [.., 2*rb] grid
    P, rows, N = 3, 32, 128
    rb = N * 2
    nb = 2

    def chunk_of(s, b):
        return [((s * nb + b) * rows * 2 * rb + (rb if b % 2 else 0), 2 * rb)], 0
    c = Case(P, nb * rows, N, rows, P * nb * rows * rb, chunk_of, dst_bytes=P * nb * rows * 2 * rb)
    # the fill writes contiguous blocks; as 2D windows they are `rows` rows of rb bytes
    c.region = lambda b: (b * rows * rb, rb, rows, rb)
    c.run(transport)


@pytest.mark.parametrize("transport", ["bulk", "copy_engines"])
def test_some_peers_with_groups_and_consumer_gather(transport):
    # every rank fills its own quarter of its buffer in four blocks; each block goes to a subset
    # of the other ranks, at its own offsets.  One group per rank holding the chunks addressed to
    # it, and one of every chunk: each rank counts only what reaches it, as the oracle does.  A
    # consumer at rank 2 reads exactly the chunks addressed to it
    P, rows, N, seed = 4, 32, 256, 91
    rb = N * 2
    B = rows * rb
    S = 4 * B
    masks = [0b0110, 0b1000, 0b0001, 0b1111]
    spec = [[masks[(s + b) % 4] for b in range(4)] for s in range(P)]
    region = lambda s, b: (s * S + b * B, B, 1, B)
    o = OP.Plan([np.zeros(P * S, dtype=np.uint8) for _ in range(P)],
                [OS.Schedule([OS.Chunk([region(s, b)], 1, peers=spec[s][b]) for b in range(4)]) for s in range(P)],
                allgather=False)
    scheds = []
    for s in range(P):
        sc = D.dtt_schedule_empty()
        for b in range(4):
            sc.add_chunk([region(s, b)], 1, peers=spec[s][b])
        scheds.append(sc)
    bufs = [torch.zeros(P * S, dtype=torch.uint8, device="cuda") for _ in range(P)]
    plan = D.Plan(bufs, P * S, scheds, _opts(transport))
    for sc in scheds:
        sc.free()
    desc = D.fill_desc("bf16", seed, 4 * rows, N, rb, P * S, [s * S for s in range(P)], rows, N, 1, 1,
                       mark_mode=D.MARK_PER_STEP)
    G = 4 * P
    groups = [[g for g in range(G) if o.owner[g] != q and q in o.chunks[g].receivers(P, o.owner[g])]
              for q in range(P)] + [list(range(G))]
    assert all(groups)
    plan.define_groups(groups)
    o.define_groups(groups)
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    out = torch.zeros(P * S, dtype=torch.uint8, device="cuda")
    status = torch.full((G,), 99, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    try:
        for R in (1, 2):
            h = plan.start(prod)
            plan.consumer_gather(2, out, 1 << 24, status, 8, cons)
            D.dtt_fill_producer(bufs, desc, h, prod)
            rep = plan.wait()
            cons.synchronize()
            assert rep.status == D.OK
            o.start()
            for s in range(P):
                o.bufs[s][s * S:(s + 1) * S] = H.fill_slice_bytes("bf16", seed, s, R, 4 * rows, N)
                for g in o.chunks_of(s):
                    o.mark_ready(s, g)
            o.copier_progress()
            assert o.wait()[0] == OP.OK
            for q in range(P):
                np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q])
            np.testing.assert_array_equal(plan.read_gates()[:, :, :5], o.gates)
            np.testing.assert_array_equal(plan.read_group_counters(), o.group_counters)
            assert status.cpu().tolist() == [0] * G
            got, want = out.cpu().numpy(), o.bufs[2]
            for g in groups[2]:
                off, n, _, _ = o.chunks[g].regions[0]
                np.testing.assert_array_equal(got[off:off + n], want[off:off + n])
            plan.next_round()
            o.next_round()
    finally:
        plan.close()


def test_destination_plans_refuse_what_needs_in_place_chunks():
    c = _reduce_scatter(P=2)
    plan, bufs, dst, desc = c.library("bulk")
    try:
        with pytest.raises(D.DttError) as e:
            plan.define_block_groups(4096)
        assert e.value.code == D.EINVAL
        with pytest.raises(D.DttError) as e:
            plan.allgather_host([None, None], None, 0, torch.cuda.current_stream())
        assert e.value.code == D.EINVAL
    finally:
        plan.close()
