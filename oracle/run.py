"""Oracle: one workload end to end -- its schedules from the oracle's builders, its producers'
writes and marks, the copier queues and wait().  TEST INFRASTRUCTURE ONLY (oracle/__init__).

``w`` is a workload description (workloads.Workload): P virtual ranks, an M x N slice per
sending rank, a schedule kind.  Each producer writes its slice for the round (oracle.hashfill)
and then marks every chunk ``writers`` times ("Triggered Plans", section Model: a round is
start(), the producer marks every chunk ready, wait()).
"""
from __future__ import annotations

import numpy as np

from . import hashfill as H
from . import plan as OP
from . import schedule as OS


def schedules(w):
    rb = w.row_bytes
    out = []
    for r in range(w.P):
        if r not in w.senders():
            out.append(OS.Schedule())
            continue
        off = w.slice_offset(r)
        if w.kind == "whole":
            out.append(OS.whole(off, w.M, rb, rb, w.num_programs))
        elif w.kind == "chunks":
            out.append(OS.chunks(off, w.M, rb, rb, w.num_chunks))
        else:
            tm, tn = -(-w.M // w.BM), -(-w.N // w.BN)
            order = (lambda s: OS.order_grouped(s, tm, tn, w.group_m)) if w.group_m else None
            out.append(OS.tile_chunks(off, w.M, w.N, w.elem_bytes, rb, w.BM, w.BN,
                                      w.tiles_per_chunk, order))
    return out


def make_plan(w, copy_data=True, initial_round=1):
    """The oracle plan of w; copy_data=False keeps gates only (large workloads)."""
    n = w.buf_bytes if copy_data else 1
    bufs = [np.zeros(n, dtype=np.uint8) for _ in range(w.P)]
    return OP.Plan(bufs, schedules(w), allgather=not w.broadcast,
                   initial_round=initial_round, validate=copy_data, copy_data=copy_data)


def run_round(o, w, marks=True):
    """Round o.round: the producers write their slices and mark every chunk; the copier
    queues run; returns wait()'s (status, short, extra)."""
    o.start()
    for r in w.senders():
        if o.copy_data:
            off = w.slice_offset(r)
            o.bufs[r][off:off + w.slice_bytes] = H.fill_slice_bytes(w.dtype, w.seed, r, o.round,
                                                                     w.M, w.N)
        if marks:
            for c in o.chunks_of(r):
                for _ in range(o.chunks[c].writers):
                    o.mark_ready(r, c)
    o.copier_progress()
    return o.wait()


def expected_bytes(w, rnd, offsets):
    """Closed form of the gathered buffers at byte offsets (the same in every rank's buffer):
    the owning rank's value for round rnd."""
    offsets = np.asarray(offsets, dtype=np.int64)
    out = np.zeros(len(offsets), dtype=np.uint8)
    e = w.elem_bytes
    S = w.slice_bytes
    owner = np.zeros(len(offsets), dtype=np.int64) if w.broadcast else offsets // S
    for r in np.unique(owner):
        sel = owner == r
        local = offsets[sel] - (0 if w.broadcast else r * S)
        rows = local // w.row_bytes
        cols = (local % w.row_bytes) // e
        vals = H.values_at(w.dtype, w.seed, int(r), rnd, rows, cols, w.N)
        raw = np.ascontiguousarray(vals).view(np.uint8).reshape(-1, e)
        out[sel] = raw[np.arange(len(local)), local % e]
    return out
