"""Helpers shared by the GPU parity tests: the oracle side of a workload (its own schedules,
its own produce step) and sampled expected values for full-size workloads."""
import numpy as np

import workloads as W
from oracle import hashfill as H
from oracle import plan as OP
from oracle import schedule as OS


def oracle_schedules(w):
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


def oracle_plan(w, copy_data=True, initial_round=1):
    n = w.buf_bytes if copy_data else 1
    bufs = [np.zeros(n, dtype=np.uint8) for _ in range(w.P)]
    return OP.Plan(bufs, oracle_schedules(w), allgather=not w.broadcast,
                   initial_round=initial_round, validate=copy_data, copy_data=copy_data)


def oracle_round(o, w, marks=True):
    """The producers of round o.round write their slices, then mark every chunk writers times;
    the copier runs; returns wait()'s result."""
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
    """Closed form of the gathered buffers at byte offsets (identical in every rank's buffer):
    the owner's value for round rnd."""
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


def sample_offsets(w, n, seed, o=None):
    """Random byte offsets plus the first and last byte of every region row span's ends."""
    rng = np.random.default_rng(seed)
    offs = [rng.integers(0, w.buf_bytes, n, dtype=np.int64)]
    if o is not None:
        ends = []
        for ch in o.chunks:
            for (off, rb, rows, pitch) in ch.regions:
                last = off + (rows - 1) * pitch + rb - 1
                ends += [off, off + rb - 1, last, last - rb + 1]
        offs.append(np.asarray(ends, dtype=np.int64))
    return np.unique(np.concatenate(offs))
