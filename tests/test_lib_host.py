"""Host-side checks of libdtt.so that need no GPU: exports, schedule builders against the
oracle's independent builders, the shared step-to-tile order, and plan validation."""
import ctypes as C
import itertools
import os
import re

import numpy as np
import pytest

from conftest import ROOT, ensure_built

ensure_built()

import device_triggered_transfers_gb300 as D  # noqa: E402
from oracle import schedule as OS  # noqa: E402


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(dtt_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert {"dtt_plan_create", "dtt_plan_start", "dtt_plan_wait", "dtt_plan_next_round",
            "dtt_plan_close", "dtt_schedule_tile_chunks", "dtt_barrier_handrolled",
            "dtt_fill_producer", "dtt_publish"} <= names
    lib = C.CDLL(D.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    for n in names:          # the binding declares a signature for every one of them
        assert n in D._SIGS, n


def _regions(s):
    return [(regs, w) for regs, w in s.chunks()]


def _oracle(s):
    return [([tuple(r) for r in c.regions], c.writers) for c in s.chunks]


@pytest.mark.parametrize("rows,rb,pitch,np_", [(4, 64, 64, 1), (7, 12, 16, 3), (1, 5, 5, 2),
                                               (3000, 1 << 20, 1 << 20, 8)])
def test_whole_matches_oracle(rows, rb, pitch, np_):
    a = D.dtt_schedule_whole(1024, rows, rb, pitch, np_)
    assert _regions(a) == _oracle(OS.whole(1024, rows, rb, pitch, np_))


@pytest.mark.parametrize("rows,rb,pitch,n", [(10, 4, 4, 4), (6, 4, 8, 3), (4096, 8192, 8192, 8),
                                             (17, 6, 6, 5), (2560, 1 << 20, 1 << 20, 2)])
def test_chunks_matches_oracle(rows, rb, pitch, n):
    a = D.dtt_schedule_chunks(96, rows, rb, pitch, n)
    assert _regions(a) == _oracle(OS.chunks(96, rows, rb, pitch, n))


CASES = [(7, 5, 2, 2, 2, 1, 0), (9, 9, 1, 4, 3, 4, 3), (300, 200, 2, 64, 48, 5, 2),
         (8000, 8064, 2, 128, 128, 148, 8), (2048, 4096, 2, 128, 128, 148, 0),
         (13, 203, 2, 8, 16, 7, 1), (100, 100, 4, 100, 100, 1, 0)]


@pytest.mark.parametrize("M,N,e,BM,BN,T,gm", CASES)
def test_tile_chunks_matches_oracle(M, N, e, BM, BN, T, gm):
    pitch = N * e + (16 if M < 50 else 0)
    tm, tn = -(-M // BM), -(-N // BN)
    a = D.dtt_schedule_tile_chunks(pitch * 2, M, N, e, pitch, BM, BN, T,
                                   D.ORDER_GROUPED if gm else D.ORDER_ROW_MAJOR, gm)
    order = (lambda s: OS.order_grouped(s, tm, tn, gm)) if gm else None
    assert _regions(a) == _oracle(OS.tile_chunks(pitch * 2, M, N, e, pitch, BM, BN, T, order))


def test_tile_chunks_with_python_order_and_bad_order():
    fn = lambda s: (s % 3, s // 3)   # column-major over a 3 x 2 tile grid  # noqa: E731
    a = D.dtt_schedule_tile_chunks(0, 6, 4, 1, 4, 2, 2, 2, order_fn=fn)
    assert _regions(a) == _oracle(OS.tile_chunks(0, 6, 4, 1, 4, 2, 2, 2, fn))
    with pytest.raises(D.DttError) as e:
        D.dtt_schedule_tile_chunks(0, 6, 4, 1, 4, 2, 2, 2, order_fn=lambda s: (0, 0))
    assert e.value.code == D.EINVAL


@pytest.mark.parametrize("tm,tn,gm", [(63, 63, 8), (5, 7, 2), (16, 32, 1), (3, 3, 5)])
def test_tile_of_matches_oracle(tm, tn, gm):
    for s in range(tm * tn):
        assert D.dtt_tile_of(D.ORDER_GROUPED, gm, s, tm, tn) == OS.order_grouped(s, tm, tn, gm)
        assert D.dtt_tile_of(D.ORDER_ROW_MAJOR, 0, s, tm, tn) == OS.order_row_major(s, tm, tn)


def test_hand_built_schedule_and_1gib_split():
    s = D.dtt_schedule_empty()
    s.add_chunk([(0, 5 * (1 << 29), 1, 5 * (1 << 29)), (100, 8, 3, 16)], 2)
    regs, w = s.chunk(0)
    assert w == 2
    assert regs == [(0, 1 << 30, 1, 1 << 30), (1 << 30, 1 << 30, 1, 1 << 30),
                    (2 << 30, 1 << 29, 1, 1 << 29), (100, 8, 3, 16)]
    with pytest.raises(D.DttError):
        s.add_chunk([(0, 8, 1, 8)], 0)


def _create(bufs_n, buf_bytes, scheds, **opts):
    o = D.dtt_plan_opts_default(**opts)
    fake = [0x10000000 * (i + 1) for i in range(bufs_n)]   # never dereferenced by validation
    try:
        D.Plan(fake, buf_bytes, scheds, o).close()
    except D.DttError as e:
        return e.code
    return D.OK


def test_plan_validation_codes_without_a_gpu():
    P, M, rb = 3, 8, 64
    S = M * rb
    good = [D.dtt_schedule_chunks(r * S, M, rb, rb, 2) for r in range(P)]
    # a valid plan passes validation and only then needs the device
    code = _create(P, P * S, good)
    assert code in (D.ECUDA, D.OK)
    bad = list(good)
    bad[1] = D.dtt_schedule_whole(0, P * M, rb, rb, 1)    # the whole buffer, not its own rows
    assert _create(P, P * S, bad) == D.EOUTOFROWS
    assert _create(P, P * S, bad, allgather=0) == D.EOVERLAP
    assert _create(P, P * S, good, max_regions=5) == D.ECAPACITY
    assert _create(P, P * S, good, host_piece_bytes=1000) == D.EINVAL
    outside = [D.dtt_schedule_whole(P * S - 8, 1, 16, 16, 1), None, None]
    assert _create(P, P * S, outside, allgather=0) == D.EINVAL
    # interleaved 2D windows that share no byte pass; shifted by one byte they overlap
    a, b, c = D.dtt_schedule_empty(), D.dtt_schedule_empty(), D.dtt_schedule_empty()
    a.add_chunk([(0, 4, 3, 8)], 1)
    b.add_chunk([(4, 4, 3, 8)], 1)
    c.add_chunk([(3, 4, 3, 8)], 1)
    assert _create(2, 24, [a, b], allgather=0) in (D.ECUDA, D.OK)
    assert _create(2, 24, [a, c], allgather=0) == D.EOVERLAP


def _i32(n):
    import torch
    return torch.zeros(n, dtype=torch.int32)


def test_reveal_wrappers_refuse_short_lists_and_tensors():
    # the reveal reads and writes P slices of `size` int32 and P status words: a short list or
    # tensor is refused on the host, before any kernel could run past it
    P, size = 4, 16
    ok = [_i32(size) for _ in range(P)]
    cases = [
        (ok, ok[:3], ok, _i32(P)),                         # data short of a slice
        (ok, ok, ok[:2], _i32(P)),                         # y short of slices
        (ok, ok, ok[:3] + [_i32(size - 1)], _i32(P)),      # one y slice too small
        (ok[:3] + [_i32(1)], ok, ok, _i32(P)),             # one x slice too small
        (ok, ok, ok, _i32(P - 1)),                         # status too small
        (ok, ok, ok, None),
    ]
    for x, data, y, status in cases:
        with pytest.raises(D.DttError) as e:
            D.dtt_barrier_reveal_noalloc(x, data, y, size, 100, status)
        assert e.value.code == D.EINVAL
    import torch
    with pytest.raises(D.DttError) as e:        # not int32
        D.dtt_barrier_reveal_noalloc(ok, ok, [torch.zeros(size, dtype=torch.int16)] * P, size, 100, _i32(P))
    assert e.value.code == D.EINVAL


def test_barrier_reveal_method_refuses_short_lists():
    b = D.Barrier.__new__(D.Barrier)      # the argument check runs before the library is called
    b._h, b.P = C.c_void_p(0), 4
    ok = [_i32(8) for _ in range(4)]
    with pytest.raises(D.DttError) as e:
        b.reveal(ok, ok[:3], ok, 8, 100, _i32(4))
    assert e.value.code == D.EINVAL


def test_handrolled_wrapper_refuses_short_windows():
    P = 4
    ok = [_i32(P) for _ in range(P)]
    for signal, y, status in [(ok, ok[:3], _i32(P)), (ok[:3] + [_i32(P - 1)], ok, _i32(P)),
                              (ok, ok, _i32(P - 1))]:
        with pytest.raises(D.DttError) as e:
            D.dtt_barrier_handrolled(signal, y, 1, 100, status)
        assert e.value.code == D.EINVAL


def test_library_grouped_order_short_last_group_golden():
    # the order the library's producers run (dtt_tile_of) against the hand-worked tables
    path = os.path.join(ROOT, "tests", "golden", "grouped_order.txt")
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        row = line.split()
        i = row.index(":")
        tiles_m, tiles_n, gm = (int(x) for x in row[:i])
        steps = [tuple(int(v) for v in t.split(",")) for t in row[i + 1:]]
        got = [D.dtt_tile_of(D.ORDER_GROUPED, gm, s, tiles_m, tiles_n) for s in range(len(steps))]
        assert got == steps


def test_binding_structs_match_the_c_header(tmp_path):
    # every struct the binding passes by pointer has the header's size and field offsets
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    structs = {"dtt_region": D.dtt_region, "dtt_dest": D.dtt_dest, "dtt_order": D.dtt_order,
               "dtt_plan_opts": D.dtt_plan_opts,
               "dtt_group_table": D.dtt_group_table, "dtt_handle": D.dtt_handle, "dtt_report": D.dtt_report, "dtt_fill_desc": D.dtt_fill_desc,
               "dtt_allreduce_desc": D.dtt_allreduce_desc}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dtt.h"', 'int main(void) {']
    for name, cls in structs.items():
        lines.append(f'printf("{name} %zu\\n", sizeof({name}));')
        for f in cls._fields_:
            lines.append(f'printf("{name}.{f[0]} %zu\\n", offsetof({name}, {f[0]}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                  check=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == C.sizeof(cls), name
        for f in cls._fields_:
            assert int(got[f"{name}.{f[0]}"]) == getattr(cls, f[0]).offset, (name, f[0])


def test_prepared_barrier_arguments_are_checked_once_at_construction():
    ok = [_i32(8) for _ in range(4)]
    with pytest.raises(D.DttError):
        D.RevealArgs(ok, ok[:3], ok, 8, _i32(4))
    with pytest.raises(D.DttError):
        D.HandrolledArgs(ok, ok, _i32(3))
    a = D.RevealArgs(ok, ok, ok, 8, _i32(4))
    assert a.P == 4 and a.size == 8
    b = D.Barrier.__new__(D.Barrier)
    b._h, b.P = C.c_void_p(0), 5
    with pytest.raises(D.DttError):            # prepared for 4 ranks, barrier of 5
        b.reveal(a)


# ---- other destinations: schedule API and plan validation against the oracle's verdicts -----------
def test_add_chunk_to_splits_contiguous_ranges_with_their_destinations():
    s = D.dtt_schedule_empty()
    G = 1 << 30
    s.add_chunk([(0, 5 * G // 2, 1, 5 * G // 2)], 1, dests=[(1000, 5 * G // 2)], peers=0b100)
    regs, w = s.chunk(0)
    dests, mask = s.dests(0)
    assert [r[1] for r in regs] == [G, G, G // 2] and [r[0] for r in regs] == [0, G, 2 * G]
    assert dests == [(1000, G), (1000 + G, G), (1000 + 2 * G, G // 2)] and mask == 0b100
    # contiguous rows landing with a wider pitch stay one 2D window
    s.add_chunk([(0, 64, 4, 64)], 2, dests=[(512, 128)])
    assert s.chunk(1) == ([(0, 64, 4, 64)], 2) and s.dests(1) == ([(512, 128)], 0)
    s.add_chunk([(0, 64, 1, 64)], 1)
    assert s.dests(2) == (None, 0)
    with pytest.raises(D.DttError):                       # destination pitch below the row bytes
        s.add_chunk([(0, 64, 4, 64)], 1, dests=[(0, 32)])
    s.free()


def _lib_verdict(P, nbytes, chunks_per_rank, dst_bytes=0):
    """Create a plan over fake (never dereferenced) buffer addresses: validation runs first, so
    an invalid plan fails before any CUDA call.  Returns the error code, or None when it passes
    validation (then creation would need a GPU, which is not tried here)."""
    scheds = []
    for r in range(P):
        s = D.dtt_schedule_empty()
        for (regs, writers, dests, peers) in chunks_per_rank[r]:
            s.add_chunk(regs, writers, dests=dests, peers=peers)
        scheds.append(s)
    opts = D.dtt_plan_opts_default(allgather=0)
    arr = (C.c_void_p * P)(*[0x100000 * (r + 1) for r in range(P)])
    if dst_bytes:
        darr = (C.c_void_p * P)(*[0x900000 * (r + 1) for r in range(P)])
        opts.dst_bufs = C.cast(darr, C.c_void_p).value
        opts.dst_bytes = dst_bytes
    sch = (C.c_void_p * P)(*[x.handle.value for x in scheds])
    out = C.c_void_p()
    rc = D.lib().dtt_plan_create(arr, nbytes, P, sch, C.byref(opts), None, C.byref(out))
    for x in scheds:
        x.free()
    if rc == D.OK:          # a device was there: release the plan (no kernel ever ran on it)
        D.lib().dtt_plan_close(out)
    return rc


def _oracle_verdict(P, nbytes, chunks_per_rank, dst_bytes=0):
    scheds = [OS.Schedule([OS.Chunk(list(regs), w, dests=dests, peers=(peers or None))
                           for (regs, w, dests, peers) in chunks_per_rank[r]]) for r in range(P)]
    try:
        OS.validate(scheds, nbytes, False, dst_bytes=dst_bytes or None)
    except OS.PlanError as e:
        return {"EOVERLAP": D.EOVERLAP, "EINVAL": D.EINVAL}[e.code]
    return None


DEST_CASES = {
    "two_copies_same_bytes": (3, 64, [[([(0, 8, 1, 8)], 1, [(40, 8)], 0b100)],
                                      [([(8, 8, 1, 8)], 1, [(44, 8)], 0b100)], []], 0),
    "onto_receivers_sent_bytes": (2, 64, [[([(0, 8, 1, 8)], 1, [(16, 8)], 0)],
                                          [([(16, 8, 1, 8)], 1, None, 0b01)]], 0),
    "separate_buffers_allow_it": (2, 64, [[([(0, 8, 1, 8)], 1, [(16, 8)], 0)],
                                          [([(16, 8, 1, 8)], 1, None, 0b01)]], 32),
    "past_the_end": (2, 64, [[([(0, 8, 1, 8)], 1, [(60, 8)], 0)], []], 0),
    "past_separate_end": (2, 64, [[([(0, 8, 1, 8)], 1, [(28, 8)], 0)], []], 32),
    "mask_outside_plan": (2, 64, [[([(0, 8, 1, 8)], 1, None, 0b100)], []], 0),
    "reduce_scatter_ok": (3, 96, [[([(b * 8, 8, 1, 8)], 1, [(48 + s * 8, 8)], 1 << b) for b in range(3) if b != s]
                                  for s in range(3)], 0),
    "pitched_rows_overlap_other": (2, 256, [[([(0, 8, 3, 16)], 1, [(100, 40)], 0)],
                                            [([(200, 8, 1, 8)], 1, [(180, 8)], 0b01)]], 0),
    "pitched_rows_interleave_ok": (3, 256, [[([(0, 8, 3, 16)], 1, [(100, 16)], 0b100)],
                                            [([(64, 8, 3, 16)], 1, [(108, 16)], 0b100)], []], 0),
}


@pytest.mark.parametrize("name", sorted(DEST_CASES))
def test_destination_validation_matches_the_oracle(name):
    P, nbytes, chunks, dst = DEST_CASES[name]
    want = _oracle_verdict(P, nbytes, chunks, dst)
    got = _lib_verdict(P, nbytes, chunks, dst)
    if want is None:
        assert got not in (D.EOVERLAP, D.EINVAL), name      # passes validation (no GPU here)
    else:
        assert got == want, (name, got, want)


def test_plan_rank_count_is_checked_before_any_device_call():
    arr = (C.c_void_p * 17)(*[0x1000 * (r + 1) for r in range(17)])
    out = C.c_void_p()
    rc = D.lib().dtt_plan_create(arr, 1 << 20, 17, None, None, None, C.byref(out))
    assert rc == D.EINVAL
    rc = D.lib().dtt_plan_create(arr, 1 << 20, 0, None, None, None, C.byref(out))
    assert rc == D.EINVAL


def test_overlap_options_are_checked_before_any_device_call():
    # overlapping rounds need the copier beside the producers: a copier ordered after them
    # (deferred_copier = 1) would leave the next round's producers waiting on nothing
    arr = (C.c_void_p * 2)(0x1000, 0x2000)
    out = C.c_void_p()
    for over in (dict(overlap=1, deferred_copier=1), dict(overlap=2)):
        opts = D.dtt_plan_opts_default(**over)
        rc = D.lib().dtt_plan_create(arr, 1 << 20, 2, None, C.byref(opts), None, C.byref(out))
        assert rc == D.EINVAL, over
        assert b"overlap" in D.lib().dtt_last_error()
    assert D.lib().dtt_plan_pending_round(None) == 0


def test_new_entry_points_refuse_a_null_plan_without_a_gpu():
    L = D.lib()
    rep = D.dtt_report()
    slices = (C.c_void_p * 2)()
    assert L.dtt_allgather_host_rounds(None, 1, slices, None, 0, None, C.byref(rep)) == D.EINVAL
    assert L.dtt_plan_next_round(None) == D.EINVAL
    assert L.dtt_plan_wait(None, C.byref(rep)) == D.EINVAL
    assert L.dtt_plan_pending_round(None) == 0


def test_schedules_from_tensor_slices_match_the_offset_builders():
    # the pages' form -- whole(mine), chunks(mine, n, base=out), tile_chunks(mine, (BM, BN), T,
    # order=..., base=out) -- gives the same regions as the offset-based builders
    import torch
    P, M, N = 4, 96, 160
    out = torch.zeros(P * M, N, dtype=torch.bfloat16)
    rb = N * 2
    for r in (0, 2, 3):
        mine = out[r * M:(r + 1) * M]
        assert _regions(D.chunks(mine, 5, base=out)) == _regions(D.dtt_schedule_chunks(r * M * rb, M, rb, rb, 5))
        assert _regions(D.whole(mine, 3, base=out)) == _regions(D.dtt_schedule_whole(r * M * rb, M, rb, rb, 3))
        got = D.tile_chunks(mine, (32, 48), 4, order=("grouped", 2), base=out)
        want = D.dtt_schedule_tile_chunks(r * M * rb, M, N, 2, rb, 32, 48, 4, D.ORDER_GROUPED, 2)
        assert _regions(got) == _regions(want)
        tm, tn = -(-M // 32), -(-N // 48)
        fn = lambda s: D.dtt_tile_of(D.ORDER_GROUPED, 2, s, tm, tn)   # the producer's own mapping
        assert _regions(D.tile_chunks(mine, (32, 48), 4, order=fn, base=out)) == _regions(want)
    # a column window: strided rows, pitch = the full row
    win = out[M:2 * M, 32:96]
    assert _regions(D.chunks(win, 3, base=out)) == \
        _regions(D.dtt_schedule_chunks(M * rb + 64, M, 128, rb, 3))
    with pytest.raises(D.DttError):
        D.chunks(out.t()[:, :8], 2, base=out)          # rows not contiguous
    with pytest.raises(D.DttError):
        D.chunks(torch.zeros(8, 8, dtype=torch.bfloat16), 2, base=out)   # not inside base


def _allreduce_create(P=2, bufs=None, buf_bytes=1 << 20, staging=None, staging_bytes=0, rs=None, ag=None, **desc):
    d = D.dtt_allreduce_desc()
    d.dtype, d.sub_blocks, d.block_rows, d.cols, d.pitch = D.BF16, 2, 64, 256, 0
    for k, v in desc.items():
        setattr(d, k, v)
    arr = (C.c_void_p * max(P, 1))(*(bufs or [0x10000 * (r + 1) for r in range(P)]))
    stg = (C.c_void_p * P)(*staging) if staging is not None else None
    out = C.c_void_p()
    rc = D.lib().dtt_allreduce_create(arr, buf_bytes, stg, staging_bytes, P, C.byref(d),
                                      C.byref(rs) if rs is not None else None,
                                      C.byref(ag) if ag is not None else None, None, None, C.byref(out))
    return rc, D.lib().dtt_last_error().decode()


@pytest.mark.parametrize("case,kw,words", [
    ("one rank", dict(P=1), "P <="),
    ("seventeen ranks", dict(P=17), "P <="),
    ("u8", dict(dtype=D.U8), "dtype"),
    ("no rows", dict(block_rows=0), "block_rows"),
    ("sub-blocks not dividing", dict(sub_blocks=3), "divide"),
    ("rows not 16-byte multiples", dict(cols=4), "multiples of 16"),
    ("pitch not a 16-byte multiple", dict(pitch=520), "multiples of 16"),
    ("pitch below the row", dict(pitch=496), "pitch >= row bytes"),
    ("reduce threads", dict(reduce_threads=100), "reduce_threads"),
    ("one warp", dict(reduce_threads=32), "reduce_threads"),
    ("buffer too small in place", dict(buf_bytes=2 * 128 * 512 - 16), "cannot hold"),
    ("staging too small", dict(staging=[0x100000, 0x200000], staging_bytes=1000), "staging buffers need"),
    ("unaligned buffer", dict(bufs=[0x10000, 0x20008]), "16-byte aligned"),
    ("rows x pitch past 64 bits", dict(pitch=1 << 60), "overflows"),
    ("more than 4096 sub-blocks", dict(P=16, block_rows=257, sub_blocks=257, buf_bytes=1 << 30), "4096 sub-blocks"),
    ("copy-engine reduce-scatter", dict(rs=D.dtt_plan_opts_default(method=2)), "copy-engine"),
    ("overlapped all-gather", dict(ag=D.dtt_plan_opts_default(overlap=1)), "overlap"),
    ("copier beside, deferred", dict(rs=D.dtt_plan_opts_default(deferred_copier=2)), "deferred_copier"),
    ("one plan in order", dict(rs=D.dtt_plan_opts_default(deferred_copier=1)), "same way"),
])
def test_allreduce_arguments_are_checked_before_any_device_call(case, kw, words):
    rc, msg = _allreduce_create(**kw)
    assert rc == D.EINVAL, (case, msg)
    assert words in msg, (case, msg)


def test_allreduce_calls_refuse_a_null_all_reduce_without_a_gpu():
    L = D.lib()
    a, b = D.dtt_report(), D.dtt_report()
    err = C.c_void_p(0x1000)
    assert L.dtt_allreduce_start(None, None, None) == D.EINVAL
    assert L.dtt_allreduce_reduce(None, err, None) == D.EINVAL
    assert L.dtt_allreduce_wait(None, C.byref(a), C.byref(b)) == D.EINVAL
    assert L.dtt_allreduce_next_round(None) == D.EINVAL
    assert L.dtt_allreduce_plans(None, None, None) == D.EINVAL
    parts = (C.c_void_p * 2)()
    assert L.dtt_allreduce_host(None, parts, None, 0, err, None, C.byref(a), C.byref(b)) == D.EINVAL
    assert L.dtt_allreduce_destroy(None) == D.OK
