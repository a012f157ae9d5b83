"""Pins for the oracle's schedule builders and plan validation (oracle/schedule.py)."""
import itertools
import os

import numpy as np
import pytest

from oracle import schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        if line.strip() and not line.startswith("#"):
            out.append(line.split())
    return out


def test_linear_split_golden():
    for row in _golden("linear_split.txt"):
        total = int(row[0])
        pieces = [int(x) for x in row[2:]]
        regs = S.split_linear(1000, total)
        assert [r[1] for r in regs] == pieces
        assert regs[0][0] == 1000
        assert all(r[2] == 1 and r[3] == r[1] for r in regs)
        assert [r[0] for r in regs] == [1000 + sum(pieces[:i]) for i in range(len(pieces))]


def test_workload_counts_golden():
    g = {row[0]: [int(x) for x in row[1:]] for row in _golden("schedule_counts.txt")}
    M, N, e = 8000, 8064, 2
    pitch = N * e
    tm, tn = -(-M // 128), -(-N // 128)
    sch = S.tile_chunks(0, M, N, e, pitch, 128, 128, 148,
                        order=lambda s: S.order_grouped(s, tm, tn, 8))
    assert sch.n_regions == g["tiles.n_tiles"][0]
    assert sch.n_chunks == g["tiles.n_chunks"][0]
    assert sch.chunks[-1].writers == g["tiles.last_chunk_steps"][0]
    assert all(c.writers == 148 for c in sch.chunks[:-1])
    regs = [r for c in sch.chunks for r in c.regions]
    assert sum(1 for r in regs if r[2] == 64) == g["tiles.edge_regions_64_rows"][0]
    assert sum(1 for r in regs if r[2] == 128) == 3969 - 63
    assert {r[1] for r in regs} == {g["tiles.row_bytes"][0]}
    assert {r[3] for r in regs} == {g["tiles.pitch"][0]}

    sch = S.tile_chunks(0, 2048, 4096, 2, 8192, 128, 128, 148)
    assert sch.n_regions == g["gemm.n_tiles"][0]
    assert [c.writers for c in sch.chunks] == g["gemm.chunk_steps"]

    sch = S.chunks(0, 4096, 8192, 8192, 8)
    assert sch.n_chunks == g["chunks.n_chunks"][0]
    assert all(c.nbytes == g["chunks.chunk_bytes"][0] and c.writers == 1 for c in sch.chunks)
    assert all(len(c.regions) == 1 and c.regions[0][2] == 1 for c in sch.chunks)


def _naive_tile_owner(M, N, BM, BN):
    """Per-element tile id by direct division (the definition of a BM x BN tiling)."""
    r = np.arange(M)[:, None] // BM
    c = np.arange(N)[None, :] // BN
    return r * (-(-N // BN)) + c


@pytest.mark.parametrize("M,N,BM,BN,T,gm", [
    (7, 5, 2, 2, 1, 0), (7, 5, 2, 2, 3, 2), (9, 9, 4, 3, 4, 3), (16, 8, 4, 4, 2, 1),
    (5, 11, 8, 4, 2, 5), (13, 6, 3, 6, 5, 2), (1, 1, 1, 1, 1, 1), (10, 10, 3, 3, 100, 4)])
def test_tile_chunks_cover_slice_exactly(M, N, BM, BN, T, gm):
    e = 2
    pitch = (N + 3) * e                    # padded rows: bytes between rows stay unsent
    base = 3 * pitch
    tm, tn = -(-M // BM), -(-N // BN)
    order = (lambda s: S.order_grouped(s, tm, tn, gm)) if gm else None
    sch = S.tile_chunks(base, M, N, e, pitch, BM, BN, T, order=order)
    nbytes = base + M * pitch
    cover = np.zeros(nbytes, dtype=np.int32)
    owner_tile = _naive_tile_owner(M, N, BM, BN)
    step = 0
    for k, ch in enumerate(sch.chunks):
        assert ch.writers == len(ch.regions)
        for reg in ch.regions:
            m = S.region_byte_mask(reg, nbytes)
            cover += m
            # the region's bytes are exactly the elements of one tile
            idx = np.nonzero(m)[0] - base
            rows, cols = idx // pitch, (idx % pitch) // e
            assert np.all(cols < N)
            assert len(np.unique(owner_tile[rows, cols])) == 1
            tile = owner_tile[rows[0], cols[0]]
            assert (owner_tile == tile).sum() * e == len(idx)
            step += 1
    assert step == tm * tn
    want = np.zeros(nbytes, dtype=np.int32)
    for r in range(M):
        want[base + r * pitch: base + r * pitch + N * e] = 1
    assert np.array_equal(cover, want)


@pytest.mark.parametrize("tiles_m,tiles_n", [(1, 1), (3, 5), (8, 8), (63, 63), (17, 4), (5, 17)])
def test_grouped_order_special_cases_and_bijection(tiles_m, tiles_n):
    T = tiles_m * tiles_n
    # GROUP_M = 1 sweeps rows in order: the row-major order
    assert [S.order_grouped(s, tiles_m, tiles_n, 1) for s in range(T)] == \
        [(s // tiles_n, s % tiles_n) for s in range(T)]
    # GROUP_M >= tiles_m makes one group of all rows: the column-major order
    assert [S.order_grouped(s, tiles_m, tiles_n, tiles_m + 3) for s in range(T)] == \
        [(s % tiles_m, s // tiles_m) for s in range(T)]
    for gm in (2, 3, 8):
        seen = {S.order_grouped(s, tiles_m, tiles_n, gm) for s in range(T)}
        assert seen == {(a, b) for a in range(tiles_m) for b in range(tiles_n)}
        # consecutive steps inside one full group go down a column of the group
        if tiles_m >= gm and tiles_n >= 2:
            assert S.order_grouped(1, tiles_m, tiles_n, gm) == (1, 0)
            assert S.order_grouped(gm, tiles_m, tiles_n, gm) == (0, 1)


def test_order_must_be_bijection():
    with pytest.raises(S.ScheduleError):
        S.tile_chunks(0, 4, 4, 1, 4, 2, 2, 1, order=lambda s: (0, 0))


def test_chunks_blocks_and_whole():
    sch = S.chunks(0, 10, 4, 4, 4)          # ceil(10/4) = 3-row blocks, last one row
    assert [c.regions for c in sch.chunks] == [[(0, 12, 1, 12)], [(12, 12, 1, 12)],
                                               [(24, 12, 1, 12)], [(36, 4, 1, 4)]]
    sch = S.chunks(100, 6, 4, 8, 3)         # strided rows: 2D windows
    assert [c.regions for c in sch.chunks] == [[(100, 4, 2, 8)], [(116, 4, 2, 8)],
                                               [(132, 4, 2, 8)]]
    w = S.whole(0, 4, 16, 16, 5)
    assert w.n_chunks == 1 and w.chunks[0].writers == 5 and w.chunks[0].regions == [(0, 64, 1, 64)]
    with pytest.raises(S.ScheduleError):
        S.chunks(0, 3, 4, 4, 4)
    with pytest.raises(S.ScheduleError):
        S.whole(0, 3, 4, 4, 0)


def test_first_chunks_global_numbering():
    scheds = [S.chunks(0, 8, 4, 4, 4), S.Schedule(), S.whole(0, 8, 4, 4, 2), S.chunks(0, 8, 4, 4, 2)]
    assert S.first_chunks(scheds) == [0, 4, 4, 5]


def test_validation_rejects_misuse():
    P, M, rb = 3, 4, 8
    buf = P * M * rb
    good = [S.chunks(r * M * rb, M, rb, rb, 2) for r in range(P)]
    S.validate(good, buf, allgather=True)
    # a schedule built from the whole buffer instead of the rank's own part
    bad = list(good)
    bad[1] = S.whole(0, P * M, rb, rb, 1)
    with pytest.raises(S.PlanError) as e:
        S.validate(bad, buf, allgather=True)
    assert e.value.code == "EOUTOFROWS"
    with pytest.raises(S.PlanError) as e:
        S.validate(bad, buf, allgather=False)
    assert e.value.code == "EOVERLAP"
    # broadcast: one sender, empty schedules elsewhere
    S.validate([S.whole(0, P * M, rb, rb, 1), S.Schedule(), S.Schedule()], buf, allgather=False)
    with pytest.raises(S.PlanError) as e:
        S.validate([S.Schedule([S.Chunk([(buf - 4, 8, 1, 8)], 1)])], buf, allgather=False)
    assert e.value.code == "EINVAL"
    with pytest.raises(S.PlanError) as e:
        S.validate(good, buf, allgather=True, max_regions=5)
    assert e.value.code == "ECAPACITY"
    # 2D windows that interleave without sharing a byte are fine
    a = S.Schedule([S.Chunk([(0, 4, 3, 8)], 1)])
    b = S.Schedule([S.Chunk([(4, 4, 3, 8)], 1)])
    S.validate([a, b], 24, allgather=False)
    c = S.Schedule([S.Chunk([(3, 4, 3, 8)], 1)])
    with pytest.raises(S.PlanError):
        S.validate([a, c], 24, allgather=False)


def _grouped_golden():
    out = []
    for row in _golden("grouped_order.txt"):
        i = row.index(":")
        tm_, tn_, gm = (int(x) for x in row[:i])
        steps = [tuple(int(v) for v in t.split(",")) for t in row[i + 1:]]
        out.append((tm_, tn_, gm, steps))
    return out


def test_grouped_order_short_last_group_golden():
    # hand-worked tables (tests/golden/grouped_order.txt): the last group of tile rows is short
    g = _grouped_golden()
    assert len(g) >= 2
    for tiles_m, tiles_n, gm, steps in g:
        assert len(steps) == tiles_m * tiles_n
        assert [S.order_grouped(s, tiles_m, tiles_n, gm) for s in range(len(steps))] == steps
