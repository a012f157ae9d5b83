"""GPU parity: the two-shot all-reduce ("Triggered Plans", Not supported yet: two-shot all-reduce,
which other destinations make possible) -- the reduce-scatter plan, the reduce kernel and the
all-gather plan of libdtt -- against the oracle's two-shot model (oracle/allreduce.py): every
byte of every buffer and staging buffer, both plans' gate words 0-4 and the reduce-scatter
plan's group counters, round after round; at full size every element against the definition;
the same for rounds fed from and returned to pinned host memory (dtt_allreduce_host)."""
import numpy as np
import pytest
import torch

from oracle import allreduce as A
from oracle import cfill
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D

SEED = 4242

COPIERS = {
    "bulk": None,   # the all-reduce's default: bulk-copy copiers, 2 CTAs x 2 x 16 KiB per SM
    "vector": dict(method=0, copier_threads=256, ctas_per_sm=1),
}


def _opts(copier, **kw):
    if COPIERS[copier] is None and not kw:
        return None
    base = dict(method=1, ctas_per_sm=2, piece_bytes=16384, stages=2) if COPIERS[copier] is None else COPIERS[copier]
    return D.dtt_plan_opts_default(**{**base, **kw})


class Case:
    def __init__(self, P, Mb, cols, J, dtype, separate=False, pitch=0, copier="bulk", reduce_ctas=0,
                 reduce_threads=0, group=1, max_polls=0, oracle=True, in_order=False, gather=True,
                 host_piece_bytes=0):
        self.P, self.Mb, self.cols, self.J, self.dtype = P, Mb, cols, J, dtype
        # the oracle's model of both plans (small cases; at full size only its layout is used)
        self.o = A.TwoShot(P, Mb, cols, dtype, J, pitch=pitch or None, separate=separate,
                           gather=gather) if oracle else None
        self.gather = gather
        _, self.pitch, self.buf_bytes, _, staging_bytes = A.layout(P, Mb, cols, dtype, pitch or None, separate)
        self.M = P * Mb
        self.Mj = Mb // J
        dev = torch.device("cuda")
        self.bufs = [torch.zeros(self.buf_bytes, dtype=torch.uint8, device=dev) for _ in range(P)]
        self.staging = [torch.zeros(staging_bytes, dtype=torch.uint8, device=dev) for _ in range(P)] \
            if separate else None
        kw = dict(max_polls=max_polls) if max_polls else {}
        if in_order:
            kw["deferred_copier"] = 1   # each kernel after its inputs (a serialising profiler's case)
        if host_piece_bytes:
            kw["host_piece_bytes"] = host_piece_bytes   # dtt_allreduce_host's least bytes a copy in
        self.ar = D.AllReduce(self.bufs, self.buf_bytes, dtype, Mb, cols, sub_blocks=J, pitch=pitch,
                              staging=self.staging, staging_bytes=staging_bytes,
                              rs_opts=_opts(copier, **kw), ag_opts=_opts(copier, **kw),
                              reduce_ctas=reduce_ctas, reduce_threads=reduce_threads, gather=gather)
        steps = self.M // self.Mj
        self.counters = torch.zeros(P * steps, dtype=torch.int32, device=dev) if group > 1 else None
        self.desc = D.fill_desc(dtype, SEED, self.M, cols, self.pitch, self.buf_bytes, [0] * P, self.Mj, cols,
                                1, 1, mark_mode=D.MARK_PER_STEP, group=group, group_counters=self.counters)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.prod = torch.cuda.Stream()
        torch.cuda.synchronize()

    def round(self, reduce_stream=None):
        h = self.ar.start(self.prod)
        if reduce_stream is not None:
            # the reduce first, on a stream of its own: its group waits order it after the
            # producers' marks and the reduce-scatter copies
            self.ar.reduce(self.err, reduce_stream)
            D.dtt_fill_producer(self.bufs, self.desc, h, self.prod)
        else:
            D.dtt_fill_producer(self.bufs, self.desc, h, self.prod)
            self.ar.reduce(self.err, self.prod)
        rs, ag = self.ar.wait()
        assert rs.status == D.OK and ag.status == D.OK   # (no all-gather plan: a zeroed report)
        torch.cuda.synchronize()       # the reduce may have run on a stream of its own
        assert int(self.err.item()) == 0

    def oracle_round(self, R):
        parts = A.hashed_partials(self.dtype, SEED, self.P, self.M, self.cols, R)
        assert self.o.round(parts) == R
        return parts

    def compare(self, what):
        for r in range(self.P):
            np.testing.assert_array_equal(self.bufs[r].cpu().numpy(), self.o.bufs[r], err_msg=f"{what} buf {r}")
            if self.staging is not None:
                np.testing.assert_array_equal(self.staging[r].cpu().numpy(), self.o.staging[r],
                                              err_msg=f"{what} staging {r}")
        np.testing.assert_array_equal(self.ar.rs.read_gates()[:, :, :5], self.o.rs.gates, err_msg=f"{what} rs gates")
        if self.gather:
            np.testing.assert_array_equal(self.ar.ag.read_gates()[:, :, :5], self.o.ag.gates, err_msg=f"{what} ag gates")
        else:
            assert self.ar.ag is None
        np.testing.assert_array_equal(self.ar.rs.read_group_counters(), self.o.rs.group_counters,
                                      err_msg=f"{what} group counters")

    def close(self):
        self.ar.close()


CASES = {
    "p2_bf16_in_place": dict(P=2, Mb=64, cols=256, J=2, dtype="bf16"),
    "p4_bf16_staging": dict(P=4, Mb=48, cols=384, J=3, dtype="bf16", separate=True),
    "p3_f32_pitched_vector": dict(P=3, Mb=40, cols=128, J=5, dtype="f32", pitch=768, copier="vector"),
    "p8_bf16": dict(P=8, Mb=16, cols=512, J=2, dtype="bf16"),
    "p4_f32_staging_vector": dict(P=4, Mb=64, cols=1024, J=4, dtype="f32", separate=True, copier="vector"),
    "p16_bf16": dict(P=16, Mb=8, cols=64, J=1, dtype="bf16"),
    "p5_bf16_one_row_sub_blocks": dict(P=5, Mb=3, cols=256, J=3, dtype="bf16"),   # 32 vectors, 152 CTAs
    "p4_bf16_few_ctas": dict(P=4, Mb=256, cols=2048, J=4, dtype="bf16", reduce_ctas=7, reduce_threads=96),
    "p6_f32_pitched_staging": dict(P=6, Mb=12, cols=36, J=4, dtype="f32", pitch=160, separate=True),
    "p4_bf16_in_order": dict(P=4, Mb=32, cols=512, J=4, dtype="bf16", in_order=True),
    "p3_f32_in_order_staging_vector": dict(P=3, Mb=20, cols=64, J=2, dtype="f32", separate=True,
                                           copier="vector", in_order=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_allreduce_matches_the_oracle(name):
    c = Case(**CASES[name])
    try:
        for R in range(1, 4):
            c.round()
            parts = c.oracle_round(R)
            c.compare(f"{name} R{R}")
            want = A.allreduce(c.dtype, parts)     # and the definition, directly
            for r in range(c.P):
                got = c.o._rows(c.bufs[r].cpu().numpy(), 0, c.M)
                assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (name, R, r)
            c.ar.next_round()
    finally:
        c.close()


SCATTER_CASES = {
    "p4_bf16_in_place": dict(P=4, Mb=48, cols=512, J=3, dtype="bf16"),
    "p3_f32_staging_vector": dict(P=3, Mb=20, cols=64, J=2, dtype="f32", separate=True, copier="vector"),
    "p5_bf16_in_order_pitched": dict(P=5, Mb=8, cols=128, J=4, dtype="bf16", pitch=320, in_order=True),
}


@pytest.mark.parametrize("name", sorted(SCATTER_CASES))
def test_reduce_scatter_matches_the_oracle(name):
    """The first shot alone (scatter_only): rank b ends with the sum over its block b and its own
    partial elsewhere; every byte of every buffer, the plan's gates and group counters."""
    c = Case(**SCATTER_CASES[name], gather=False)
    try:
        for R in range(1, 4):
            c.round()
            parts = c.oracle_round(R)
            c.compare(f"{name} R{R}")
            want = A.reduce_scatter(c.dtype, parts, c.P, c.Mb)
            for r in range(c.P):
                got = c.o._rows(c.bufs[r].cpu().numpy(), 0, c.M)
                assert np.array_equal(got.view(np.uint8), want[r].view(np.uint8)), (name, R, r)
            c.ar.next_round()
    finally:
        c.close()


def test_allreduce_reduce_launched_first_on_its_own_stream():
    c = Case(P=4, Mb=64, cols=512, J=4, dtype="bf16", group=8)
    side = torch.cuda.Stream()
    try:
        for R in range(1, 3):
            c.round(reduce_stream=side)
            c.oracle_round(R)
            c.compare(f"reduce first R{R}")
            c.ar.next_round()
    finally:
        c.close()


FULL = {
    # the benchmark's launch: 128 MiB per rank (the 4-rank chunked all-gather's size), blocks of
    # 4096 rows in 8 MiB sub-blocks; and the same in 4 MiB sub-blocks
    "p4_bf16": dict(P=4, Mb=4096, cols=4096, J=4, dtype="bf16", group=38),
    "p4_bf16_8_sub_blocks": dict(P=4, Mb=4096, cols=4096, J=8, dtype="bf16", group=38),
    "p4_f32": dict(P=4, Mb=4096, cols=2048, J=8, dtype="f32", group=38),
    # eight ranks of 128 MiB (2 GiB of buffers with the slots)
    "p8_bf16": dict(P=8, Mb=2048, cols=4096, J=4, dtype="bf16", group=19),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_allreduce_full_size_every_element(name):
    """Full-size vectors (128 MiB per rank), the producer a group of CTAs per rank: every element
    of every rank's result against the definition, two rounds; the expected sums built block by
    block from the oracle's C restatement of the producer's values."""
    f = FULL[name]
    P, Mb, cols, dtype = f["P"], f["Mb"], f["cols"], f["dtype"]
    c = Case(P=P, Mb=Mb, cols=cols, J=f["J"], dtype=dtype, group=f["group"], oracle=False)
    eb = 2 if dtype == "bf16" else 4
    view = np.uint16 if dtype == "bf16" else np.float32
    try:
        for R in range(1, 3):
            c.round()
            rb = cols * eb
            for b in range(P):
                parts = []
                for s in range(P):
                    raw = np.empty(Mb * rb, dtype=np.uint8)
                    cfill.fill_rows_into(raw, dtype, SEED, s, R, cols, b * Mb, (b + 1) * Mb)
                    parts.append(raw.view(view).reshape(Mb, cols))
                want = A.allreduce(dtype, parts).view(np.uint8).reshape(-1)
                for r in range(P):
                    got = c.bufs[r][b * Mb * rb:(b + 1) * Mb * rb].cpu().numpy()
                    np.testing.assert_array_equal(got, want, err_msg=f"{name} R{R} block {b} at rank {r}")
            c.ar.next_round()
    finally:
        c.close()


HOST_CASES = {
    "p4_bf16_in_place": dict(P=4, Mb=64, cols=256, J=2, dtype="bf16"),
    "p3_f32_pitched_staging": dict(P=3, Mb=40, cols=128, J=5, dtype="f32", pitch=768, separate=True),
    "p5_bf16_one_row_sub_blocks": dict(P=5, Mb=3, cols=256, J=3, dtype="bf16"),
    "p8_bf16_vector_copier": dict(P=8, Mb=16, cols=512, J=2, dtype="bf16", copier="vector"),
    "p2_f32_large_sub_blocks": dict(P=2, Mb=1024, cols=1024, J=2, dtype="f32"),   # 4 MiB sub-blocks
    # 8 KiB sub-blocks, copies in of at least 12 KiB a rank: two sub-blocks a step, and with
    # three sub-blocks a block a ragged last step of one
    "p4_bf16_two_sub_blocks_a_step": dict(P=4, Mb=64, cols=256, J=4, dtype="bf16", host_piece_bytes=12288),
    "p3_f32_ragged_steps_pitched": dict(P=3, Mb=48, cols=128, J=3, dtype="f32", pitch=640,
                                        host_piece_bytes=12288),
    "p16_bf16_one_sub_block_a_step": dict(P=16, Mb=8, cols=512, J=2, dtype="bf16", host_piece_bytes=4096),
}


def _pinned(arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1).copy()).pin_memory()


@pytest.mark.parametrize("name", sorted(HOST_CASES))
def test_allreduce_host_round_matches_the_oracle(name):
    """dtt_allreduce_host: the vectors from pinned host memory, the result of a different rank
    copied back each round -- every byte of every buffer and staging buffer, both plans' gates
    and the group counters against the oracle's round, and the copied-back result against the
    definition, three rounds."""
    c = Case(**HOST_CASES[name])
    eb = A.ELEM_BYTES[c.dtype]
    try:
        for R in range(1, 4):
            parts = A.hashed_partials(c.dtype, SEED, c.P, c.M, c.cols, R)
            out = torch.zeros(c.M * c.cols * eb, dtype=torch.uint8).pin_memory()
            rs, ag = c.ar.host_round([_pinned(x) for x in parts], c.err, host_out=out,
                                     out_rank=(R - 1) % c.P, stream=c.prod)
            assert rs.status == D.OK and ag.status == D.OK
            torch.cuda.synchronize()
            assert int(c.err.item()) == 0
            assert c.o.round(parts) == R
            c.compare(f"{name} R{R}")
            want = A.allreduce(c.dtype, parts)
            np.testing.assert_array_equal(out.numpy(), want.view(np.uint8).reshape(-1), err_msg=f"{name} R{R}")
    finally:
        c.close()


def test_allreduce_host_round_with_a_rank_as_it_stands_and_no_copy_back():
    """A NULL host vector leaves that rank's device vector as it stands; without host_out the
    result stays on the device; a host round and an ordinary round alternate."""
    c = Case(P=4, Mb=32, cols=512, J=4, dtype="bf16")
    S = c.M * c.cols * 2
    try:
        for R in range(1, 5):
            if R == 3:
                c.round()                              # an ordinary round between host rounds
                c.oracle_round(R)
                c.compare(f"R{R}")
                c.ar.next_round()
                continue
            parts = A.hashed_partials(c.dtype, SEED, c.P, c.M, c.cols, R)
            c.bufs[2][:S].copy_(torch.from_numpy(parts[2].view(np.uint8).reshape(-1).copy()))
            torch.cuda.synchronize()
            host = [_pinned(x) for x in parts]
            host[2] = None
            out = torch.zeros(S, dtype=torch.uint8).pin_memory() if R == 4 else None
            rs, ag = c.ar.host_round(host, c.err, host_out=out, out_rank=2, stream=c.prod)
            assert rs.status == D.OK and ag.status == D.OK
            torch.cuda.synchronize()
            assert int(c.err.item()) == 0
            assert c.o.round(parts) == R
            c.compare(f"R{R}")
            if out is not None:
                np.testing.assert_array_equal(out.numpy(), A.allreduce(c.dtype, parts).view(np.uint8).reshape(-1))
    finally:
        c.close()


def test_allreduce_host_round_refusals():
    """Host buffers too short or on the device, a wrong count and an out-of-range out_rank are
    refused before anything starts; the all-reduce stays usable."""
    c = Case(P=2, Mb=16, cols=256, J=2, dtype="bf16")
    S = c.M * c.cols * 2
    try:
        good = [torch.zeros(S, dtype=torch.uint8).pin_memory() for _ in range(2)]
        for bad in ([good[0]], [good[0], torch.zeros(S - 2, dtype=torch.uint8).pin_memory()],
                    [good[0], torch.zeros(S, dtype=torch.uint8, device="cuda")]):
            with pytest.raises(D.DttError) as ei:
                c.ar.host_round(bad, c.err, stream=c.prod)
            assert ei.value.code == D.EINVAL
        with pytest.raises(D.DttError) as ei:
            c.ar.host_round(good, c.err, out_rank=2, stream=c.prod)
        assert ei.value.code == D.EINVAL
        c.round()
        c.oracle_round(1)
        c.compare("after the refusals")
    finally:
        c.close()
    # the in-order form (the reduce could not overlap the copies in) and a reduce-scatter (no
    # all-gather plan to deliver a result) are refused too
    for kw in (dict(in_order=True), dict(gather=False)):
        c = Case(P=2, Mb=16, cols=256, J=2, dtype="bf16", **kw)
        try:
            host = [torch.zeros(S, dtype=torch.uint8).pin_memory() for _ in range(2)]
            with pytest.raises(D.DttError) as ei:
                c.ar.host_round(host, c.err, stream=c.prod)
            assert ei.value.code == D.EINVAL, kw
            c.round()
            c.oracle_round(1)
            c.compare(f"after the refusal {kw}")
        finally:
            c.close()


def test_allreduce_host_round_full_size():
    """The benchmark's all-reduce (P = 4, bf16 [16384, 4096] per rank, 4 sub-blocks of 8 MiB a
    block) from pinned host memory, two rounds: the copied-back result and every rank's device
    vector against the definition, element by element."""
    P, Mb, cols, J = 4, 4096, 4096, 4
    c = Case(P=P, Mb=Mb, cols=cols, J=J, dtype="bf16", oracle=False)
    M, rb = P * Mb, cols * 2
    try:
        for R in range(1, 3):
            host = []
            for s in range(P):
                h = torch.empty(M * rb, dtype=torch.uint8).pin_memory()
                cfill.fill_rows_into(h.numpy(), "bf16", SEED, s, R, cols, 0, M)
                host.append(h)
            out = torch.zeros(M * rb, dtype=torch.uint8).pin_memory()
            rs, ag = c.ar.host_round(host, c.err, host_out=out, out_rank=R % P, stream=c.prod)
            assert rs.status == D.OK and ag.status == D.OK
            torch.cuda.synchronize()
            assert int(c.err.item()) == 0
            for b in range(P):
                sl = slice(b * Mb * rb, (b + 1) * Mb * rb)
                parts = [host[s].numpy()[sl].view(np.uint16) for s in range(P)]
                want = A.allreduce("bf16", parts).view(np.uint8)
                np.testing.assert_array_equal(out.numpy()[sl], want, err_msg=f"R{R} block {b} copied back")
                for r in range(P):
                    np.testing.assert_array_equal(c.bufs[r][sl].cpu().numpy(), want,
                                                  err_msg=f"R{R} block {b} at rank {r}")
    finally:
        c.close()


def test_allreduce_missing_mark_fails_the_round_and_counts_the_reduce_wait():
    """One reduce-scatter chunk never marked (the producers of the other chunks run): the
    group of its sub-block never completes, the reduce's CTAs give up after the plan's poll
    limit and count it, the all-gather chunks they did not reach stay unmarked, and both waits
    fail.  Bounded waits only: nothing spins past its limit."""
    P, Mb, cols, J = 3, 8, 256, 2
    c = Case(P=P, Mb=Mb, cols=cols, J=J, dtype="bf16", max_polls=2000)
    try:
        h = c.ar.start(c.prod)
        # rank 1 writes nothing and marks every chunk but (b = 2, j = 1); the others fill
        c.desc.rank_mask = 0b101
        D.dtt_fill_producer(c.bufs, c.desc, h, c.prod)
        first = c.ar.rs.info()[1][1]
        D.dtt_publish(h, first, P * J - 1, 0, c.prod)
        c.ar.reduce(c.err, c.prod)
        rs, ag = c.ar.wait(raise_on_error=False)
        assert rs.status == D.ETIMEDOUT and ag.status == D.ETIMEDOUT
        torch.cuda.synchronize()
        assert int(c.err.item()) > 0
        # the reduce-scatter short chunk is rank 1's last; the all-gather chunks of block 2
        # from sub-block 1 on were never marked
        assert first + P * J - 1 in list(rs.short_chunks[:rs.n_short])
        ag_first = c.ar.ag.info()[1]
        assert ag_first[2] + 1 in list(ag.short_chunks[:ag.n_short])
    finally:
        c.close()


def test_allreduce_200_rounds_counters_and_gates_stay_exact():
    """Many rounds in a row: the reduce kernel's per-sub-block counters return to zero after
    every launch and both plans' gates keep counting, so round 200 matches the oracle exactly."""
    c = Case(P=3, Mb=16, cols=256, J=4, dtype="bf16")
    try:
        for R in range(1, 201):
            c.round()
            parts = c.oracle_round(R)
            if R in (1, 2, 57, 128, 200):
                c.compare(f"stress R{R}")
                want = A.allreduce("bf16", parts)
                for r in range(c.P):
                    got = c.o._rows(c.bufs[r].cpu().numpy(), 0, c.M)
                    assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (R, r)
            c.ar.next_round()
    finally:
        c.close()


def test_allreduce_round_limit():
    """Both plans start two rounds below the limit (initial_round = 2^32 - 2): two rounds run, and
    the next next_round is refused (EROUNDLIMIT), as the oracle's plans refuse it."""
    P, Mb, cols, J = 2, 8, 128, 2
    first = (1 << 32) - 2
    o = A.TwoShot(P, Mb, cols, "bf16", J, initial_round=first)
    dev = torch.device("cuda")
    bufs = [torch.zeros(o.buf_bytes, dtype=torch.uint8, device=dev) for _ in range(P)]
    opts = D.dtt_plan_opts_default(method=1, ctas_per_sm=3, piece_bytes=16384, stages=2, initial_round=first)
    ar = D.AllReduce(bufs, o.buf_bytes, "bf16", Mb, cols, sub_blocks=J, rs_opts=opts, ag_opts=opts)
    desc = D.fill_desc("bf16", SEED, P * Mb, cols, cols * 2, o.buf_bytes, [0] * P, Mb // J, cols, 1, 1)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    prod = torch.cuda.Stream()
    try:
        for R in (first, first + 1):
            h = ar.start(prod)
            D.dtt_fill_producer(bufs, desc, h, prod)
            ar.reduce(err, prod)
            rs, ag = ar.wait()
            assert rs.status == D.OK and ag.status == D.OK and rs.round == R
            parts = A.hashed_partials("bf16", SEED, P, P * Mb, cols, R)
            if R == first:
                assert o.round(parts) == R
            else:
                # the oracle's round ends with next_round, refused at the limit once the
                # round's data is final
                with pytest.raises(OP.RoundLimitError):
                    o.round(parts)
            for q in range(P):
                np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"R{R} buf {q}")
            if R == first:
                ar.next_round()
        with pytest.raises(D.DttError) as e:
            ar.next_round()
        assert e.value.code == D.EROUNDLIMIT
    finally:
        ar.close()


def test_allreduce_plans_sharing_one_copy_stream():
    """Both plans' copiers on one copy stream (plans may share a queue): the all-gather copier
    runs only after the reduce-scatter copier, which needs nothing from it, so the round still
    completes -- with less overlap -- and matches the oracle."""
    P, Mb, cols, J = 4, 32, 512, 4
    o = A.TwoShot(P, Mb, cols, "bf16", J)
    dev = torch.device("cuda")
    bufs = [torch.zeros(o.buf_bytes, dtype=torch.uint8, device=dev) for _ in range(P)]
    shared = torch.cuda.Stream(priority=-1)
    ar = D.AllReduce(bufs, o.buf_bytes, "bf16", Mb, cols, sub_blocks=J, rs_copy_stream=shared, ag_copy_stream=shared)
    desc = D.fill_desc("bf16", SEED, P * Mb, cols, cols * 2, o.buf_bytes, [0] * P, Mb // J, cols, 1, 1)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    prod = torch.cuda.Stream()
    try:
        for R in (1, 2, 3):
            h = ar.start(prod)
            D.dtt_fill_producer(bufs, desc, h, prod)
            ar.reduce(err, prod)
            rs, ag = ar.wait()
            assert rs.status == D.OK and ag.status == D.OK
            o.round(A.hashed_partials("bf16", SEED, P, P * Mb, cols, R))
            for q in range(P):
                np.testing.assert_array_equal(bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"R{R} buf {q}")
            ar.next_round()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    finally:
        ar.close()


def test_allreduce_many_one_row_sub_blocks():
    """256 sub-blocks of one row each (P = 4, 64 rows per block): the reduce's publisher reads the
    groups eight ahead, so many batches; every byte against the oracle."""
    c = Case(P=4, Mb=64, cols=512, J=64, dtype="bf16")
    try:
        for R in (1, 2):
            c.round()
            c.oracle_round(R)
            c.compare(f"256 sub-blocks R{R}")
            c.ar.next_round()
    finally:
        c.close()


def test_allreduce_producer_marks_last_to_first():
    """Each rank's partial written first, its reduce-scatter chunks then marked one by one from
    the last to the first (one publish launch per chunk): the copier's queues keep schedule order
    and the reduce takes the sub-blocks in order, so it waits for the last marks -- slower, still
    the oracle's result."""
    P, Mb, cols, J = 3, 16, 256, 4
    c = Case(P=P, Mb=Mb, cols=cols, J=J, dtype="bf16")
    try:
        for R in (1, 2):
            h = c.ar.start(c.prod)
            # the partials copied in (the fill would mark as it writes), then the marks
            parts = A.hashed_partials("bf16", SEED, P, P * Mb, cols, R)
            with torch.cuda.stream(c.prod):
                for r in range(P):
                    c.bufs[r][:P * Mb * cols * 2].copy_(torch.from_numpy(parts[r].view(np.uint8).reshape(-1)),
                                                        non_blocking=False)
            n_rank = P * J
            for r in range(P):
                first = c.ar.rs.info()[1][r]
                for k in reversed(range(n_rank)):
                    D.dtt_publish(h, first + k, 1, 0, c.prod)
            c.ar.reduce(c.err, c.prod)
            rs, ag = c.ar.wait()
            assert rs.status == D.OK and ag.status == D.OK
            c.oracle_round(R)
            c.compare(f"reversed marks R{R}")
            c.ar.next_round()
        torch.cuda.synchronize()
        assert int(c.err.item()) == 0
    finally:
        c.close()
