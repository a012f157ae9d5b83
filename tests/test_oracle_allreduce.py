"""Pins of the two-shot all-reduce oracle (oracle/allreduce.py) against what the arithmetic
fixes, not against the oracle itself: hand-worked sums (tests/golden/allreduce_sums.txt), closed
forms, the error bound of f32 summation against the exact sum, a brute-force check of the bf16
rounding against an independent nearest-even rounding, and the protocol (two plans and the
reduce step on the oracle's plan model) against the plain definition."""
import os

import numpy as np
import pytest

from oracle import allreduce as A
from oracle import hashfill as H
from oracle import plan as OP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "allreduce_sums.txt")


def _golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, rest = line.split(":")
        dtype, P = head.split()
        xs, y = rest.split("->")
        cases.append((dtype, int(P), [int(v, 16) for v in xs.split()], int(y, 16)))
    return cases


def _storage(dtype, bits):
    if dtype == "bf16":
        return np.array(bits, dtype=np.uint16)
    return np.array(bits, dtype=np.uint32).view(np.float32)


def _bits(dtype, vals):
    return np.asarray(vals).view(np.uint16 if dtype == "bf16" else np.uint32)


@pytest.mark.parametrize("case", _golden(), ids=lambda c: f"{c[0]}-P{c[1]}-{'_'.join(f'{v:x}' for v in c[2])}")
def test_golden_sums(case):
    dtype, P, xs, y = case
    assert len(xs) == P
    parts = [_storage(dtype, [x]) for x in xs]
    assert int(_bits(dtype, A.allreduce(dtype, parts))[0]) == y


def test_golden_file_covers_order_and_final_rounding():
    cases = _golden()
    assert {c[0] for c in cases} == {"bf16", "f32"} and len(cases) >= 10


def _f32_to_storage(dtype, v):
    v = np.asarray(v, dtype=np.float32)
    return H.f32_to_bf16_bits(v) if dtype == "bf16" else v


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_integer_inputs_closed_form(dtype, P):
    # x_r = r + 1 everywhere: every partial sum is a small integer, exact in f32 and bf16
    parts = [_f32_to_storage(dtype, np.full(37, r + 1.0)) for r in range(P)]
    y = A.to_f32(dtype, A.allreduce(dtype, parts))
    assert np.all(y == P * (P + 1) / 2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_opposites_cancel_to_plus_zero(dtype):
    v = H.fill_slice(dtype, 5, 0, 1, 8, 64).reshape(-1)
    neg = (_bits(dtype, v) ^ (0x8000 if dtype == "bf16" else 0x80000000)).view(v.dtype)
    zero = np.zeros_like(v)
    for parts in ([v, neg], [v, neg, zero, zero]):
        assert np.all(_bits(dtype, A.allreduce(dtype, parts)) == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_rank_is_the_identity(dtype):
    v = H.fill_slice(dtype, 9, 3, 2, 16, 32)
    assert np.array_equal(_bits(dtype, A.allreduce(dtype, [v])), _bits(dtype, v))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_error_bound_against_the_exact_sum(dtype, P):
    """Recursive f32 summation of P terms is within gamma_{P-1} * sum|x_i| of the exact sum
    (u = 2^-24, gamma_n = n u / (1 - n u)); rounding that to bf16 adds at most 2^-8 of its
    magnitude.  Values: the hashed uniforms times scales 2^-6..2^6, so terms differ in size."""
    rng = np.random.default_rng(1000 + P)
    parts, absum = [], 0
    for r in range(P):
        u = A.to_f32(dtype, H.fill_slice(dtype, 21, r, 1, 64, 128)).astype(np.float64)
        scale = 2.0 ** rng.integers(-6, 7, size=u.shape)
        parts.append(_f32_to_storage(dtype, u * scale))
    S = A.exact_sum(dtype, parts)
    absum = sum(np.abs(A.to_f32(dtype, x).astype(np.float64)) for x in parts)
    u32 = 2.0 ** -24
    gamma = (P - 1) * u32 / (1 - (P - 1) * u32)
    y = A.to_f32(dtype, A.allreduce(dtype, parts)).astype(np.float64)
    bound = gamma * absum
    if dtype == "bf16":
        bound = bound + 2.0 ** -8 * (np.abs(S) + gamma * absum)
    assert np.all(np.abs(y - S) <= bound)
    # and the bound is not vacuous: it is far below one term's size
    assert np.median(bound / np.maximum(absum, 1e-30)) < (2.0 ** -7 if dtype == "bf16" else 2.0 ** -20)


def _rne_bf16_independent(v: float) -> int:
    """Nearest bf16 to the float64 value v (ties to the even pattern), found by comparing the
    two bf16 neighbours of v exactly in float64 -- a different method from the oracle's
    bit-carry rounding."""
    if v == 0:
        return 0x8000 if np.signbit(v) else 0
    f = np.float32(v)
    assert float(f) == v            # the test only feeds values exact in f32
    hi16 = int(np.array([f]).view(np.uint32)[0]) >> 16
    lo = np.array([hi16 << 16], dtype=np.uint32).view(np.float32)[0]
    up = np.array([(hi16 + 1) << 16], dtype=np.uint32).view(np.float32)[0]
    dlo, dup = abs(v - float(lo)), abs(float(up) - v)
    if dlo < dup:
        return hi16
    if dup < dlo:
        return hi16 + 1
    return hi16 if hi16 % 2 == 0 else hi16 + 1


def test_bf16_pairs_brute_force():
    """P = 2 over bf16 values of exponents 2^-3..2^3 with every 7-bit mantissa of a stride and
    both signs: the f32 sum of two such values is exact, so y must be the nearest-even bf16 of
    the exact sum."""
    vals = []
    for e in range(124, 131):
        for m in range(0, 128, 9):
            for sgn in (0, 1):
                vals.append((sgn << 15) | (e << 7) | m)
    vals = np.array(vals, dtype=np.uint16)
    a = np.repeat(vals, len(vals))
    b = np.tile(vals, len(vals))
    y = A.allreduce("bf16", [a, b])
    exact = H.bf16_bits_to_f32(a).astype(np.float64) + H.bf16_bits_to_f32(b).astype(np.float64)
    want = np.array([_rne_bf16_independent(float(v)) for v in exact], dtype=np.uint16)
    assert np.array_equal(y, want)


def _blocks_of(P, Mb, x):
    return [x[b * Mb:(b + 1) * Mb] for b in range(P)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P,J,separate", [(2, 1, False), (3, 2, True), (4, 4, False), (4, 2, True), (8, 1, False)])
def test_two_shot_protocol_equals_the_definition(dtype, P, J, separate):
    Mb, cols = 4, 24
    o = A.TwoShot(P, Mb, cols, dtype, J, separate=separate)
    for R in range(1, 4):
        partials = A.hashed_partials(dtype, 33, P, P * Mb, cols, R)
        assert o.round(partials) == R
        want = A.allreduce(dtype, partials)
        for r in range(P):
            assert np.array_equal(_bits(dtype, o.result(r)), _bits(dtype, want)), (R, r)
        # slot s at rank b holds rank s's partial of block b (its own slot stays untouched)
        for b in range(P):
            for s in range(P):
                got = o._rows(o.stage(b), o.slot_off + s * Mb * o.pitch, Mb)
                if s == b:
                    assert not np.any(_bits(dtype, got))
                else:
                    assert np.array_equal(_bits(dtype, got), _bits(dtype, _blocks_of(P, Mb, partials[s])[b]))
        # every group is complete at its block's owner, R times over
        for b in range(P):
            for j in range(J):
                assert int(o.rs.group_counters[b, b * J + j]) == R * P
        # all-gather chunks arrived at every other rank
        for b in range(P):
            for j in range(J):
                c = o.ag.first[b] + j
                for q in range(P):
                    if q != b:
                        assert int(o.ag.gates[q, c, OP.ARRIVAL]) == R


def test_pitch_padding_is_left_alone():
    P, Mb, cols, J = 3, 4, 8, 2
    o = A.TwoShot(P, Mb, cols, "bf16", J, pitch=cols * 2 + 32)
    o.round(A.hashed_partials("bf16", 2, P, P * Mb, cols, 1))
    for r in range(P):
        for i in range(P * Mb):
            pad = o.bufs[r][i * o.pitch + cols * 2:(i + 1) * o.pitch]
            assert not np.any(pad)


def test_reduce_before_its_group_is_complete_is_refused():
    P, Mb, cols, J = 3, 2, 8, 1
    o = A.TwoShot(P, Mb, cols, "f32", J)
    o.rs.start()
    o.ag.start()
    parts = A.hashed_partials("f32", 4, P, P * Mb, cols, 1)
    for s in range(P):
        o._put_rows(o.bufs[s], 0, parts[s])
        for c in o.rs.chunks_of(s):
            if not (s == 2 and c == o.rs.first[s] + 0):   # rank 2 leaves its block-0 chunk unmarked
                o.rs.mark_ready(s, c)
    o.rs.copier_progress()
    with pytest.raises(OP.StateError):
        o.reduce_chunk(0, 0)
    o.reduce_chunk(1, 0)      # block 1 has everything


def test_schedules_and_groups_by_hand():
    """P = 2, Mb = 4 rows of 8 bytes, J = 2, in place (slots from byte 64): rank 0's chunks are
    rows 0-1 and 2-3 (block 0, only to itself), rows 4-5 and 6-7 (block 1, to rank 1's slot 0 at
    bytes 64 and 80); rank 1's block-0 chunks land in rank 0's slot 1 at bytes 96 and 112."""
    rs = A.reduce_scatter_schedules(2, 4, 2, 8, 8, 64)
    c0 = rs[0].chunks
    assert [ch.regions[0] for ch in c0] == [(0, 8, 2, 8), (16, 8, 2, 8), (32, 8, 2, 8), (48, 8, 2, 8)]
    assert [ch.dests[0][0] for ch in c0] == [64, 80, 64, 80]
    assert [ch.peers for ch in c0] == [1, 1, 2, 2]
    c1 = rs[1].chunks
    assert [ch.dests[0][0] for ch in c1] == [96, 112, 96, 112]
    assert [ch.peers for ch in c1] == [1, 1, 2, 2]
    assert A.reduce_groups(2, 2) == [[0, 4], [1, 5], [2, 6], [3, 7]]
    ag = A.allgather_schedules(2, 4, 2, 8, 8)
    assert [len(s.chunks) for s in ag] == [2, 2]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P,J,separate", [(2, 2, False), (4, 1, True), (3, 3, False)])
def test_reduce_scatter_leaves_the_other_blocks_alone(dtype, P, J, separate):
    """The first shot alone: rank b holds the sum of block b and its own partial elsewhere; the
    slots hold the peers' partials as in the all-reduce; no all-gather plan."""
    Mb, cols = 6, 16
    o = A.TwoShot(P, Mb, cols, dtype, J, separate=separate, gather=False)
    assert o.ag is None
    for R in (1, 2):
        parts = A.hashed_partials(dtype, 8, P, P * Mb, cols, R)
        o.round(parts)
        want = A.reduce_scatter(dtype, parts, P, Mb)
        y = A.allreduce(dtype, parts)
        for r in range(P):
            got = o.result(r)
            assert np.array_equal(_bits(dtype, got), _bits(dtype, want[r]))
            # block r is the sum; every other block is rank r's own partial
            assert np.array_equal(_bits(dtype, got[r * Mb:(r + 1) * Mb]), _bits(dtype, y[r * Mb:(r + 1) * Mb]))
            for b in range(P):
                if b != r:
                    assert np.array_equal(_bits(dtype, got[b * Mb:(b + 1) * Mb]),
                                          _bits(dtype, parts[r][b * Mb:(b + 1) * Mb]))


def _threaded_two_shot_round(o, parts, rng, max_polls=200000):
    """One round of the two plans with threads in every role: a producer per rank (its partial
    written and marked chunk by chunk, in a random order), a copier per (source, peer) queue of
    each plan, and a reducer per sub-block that waits on its group, adds and marks.  Gate and
    counter updates under one lock (the atomics); random short sleeps vary the interleaving."""
    import threading
    import time
    lock = threading.Lock()
    timeouts = []
    R = o.rs.start()
    assert o.ag.start() == R
    P, J, Mj = o.P, o.J, o.Mj

    def nap():
        time.sleep(float(rng.uniform(0, 2e-4)))

    def producer(s, order):
        for c in order:
            k = c - o.rs.first[s]
            b, j = divmod(k, J)
            row0 = b * o.Mb + j * Mj
            nap()
            o._put_rows(o.bufs[s], row0 * o.pitch, np.asarray(parts[s])[row0:row0 + Mj])
            with lock:
                o.rs.mark_ready(s, c)

    def copier(plan, s, p):
        for c in plan.chunks_of(s):
            if p not in plan.chunks[c].receivers(plan.P, s):
                continue
            for _ in range(max_polls):
                with lock:
                    if plan.gate_open(c):
                        break
                time.sleep(1e-5)
            else:
                timeouts.append((id(plan), s, p, c))
                return
            nap()
            ch = plan.chunks[c]
            for i, reg in enumerate(ch.regions):
                OP.copy_region(plan.bufs[s], plan.dst[p], reg, ch.dest_region(i))
            with lock:
                plan.signal_arrival(s, p, c)

    def reducer(b, j):
        for _ in range(max_polls):
            with lock:
                if o.rs.group_ready(b, b * J + j):
                    break
            time.sleep(1e-5)
        else:
            timeouts.append(("reduce", b, j))
            return
        nap()
        with lock:
            o.reduce_chunk(b, j)

    threads = []
    for s in range(P):
        order = list(o.rs.chunks_of(s))
        rng.shuffle(order)
        threads.append(threading.Thread(target=producer, args=(s, order)))
        for p in range(P):
            if p != s:
                threads.append(threading.Thread(target=copier, args=(o.rs, s, p)))
                threads.append(threading.Thread(target=copier, args=(o.ag, s, p)))
    for b in range(P):
        for j in range(J):
            threads.append(threading.Thread(target=reducer, args=(b, j)))
    rng.shuffle(threads)
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not timeouts, timeouts
    for pl in (o.rs, o.ag):
        assert pl.wait()[0] == OP.OK
        pl.next_round()
    return R


@pytest.mark.parametrize("seed", range(6))
def test_two_shot_with_threads_in_every_role(seed):
    """Producers marking in random orders, every copier queue and every reducer on threads: the
    group waits alone keep the reduce after every part has landed and the all-gather off the
    rows the reduce-scatter still reads, so every rank ends with the definition's sum."""
    rng = np.random.default_rng(seed)
    P, Mb, cols, J = (2, 3, 4, 4, 3, 2)[seed], 4, 16, (1, 2, 2, 4, 1, 2)[seed]
    dtype = "bf16" if seed % 2 == 0 else "f32"
    o = A.TwoShot(P, Mb, cols, dtype, J, separate=seed % 3 == 0)
    for R in (1, 2):
        parts = A.hashed_partials(dtype, 60 + seed, P, P * Mb, cols, R)
        assert _threaded_two_shot_round(o, parts, rng) == R
        want = A.allreduce(dtype, parts)
        for r in range(P):
            assert np.array_equal(_bits(dtype, o.result(r)), _bits(dtype, want)), (seed, R, r)
