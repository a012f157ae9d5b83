"""Glue from a workload description (workloads.py) to library calls: the schedules from the
library's builders, the plan, the fill producer's description, and one round of the path.

Everything here is argument marshalling; the work runs in libdtt.so's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

from . import (MARK_AT_END, MARK_PER_STEP, ORDER_GROUPED, ORDER_ROW_MAJOR, Plan, Schedule,
               dtt_fill_producer, dtt_plan_opts_default, dtt_schedule_chunks,
               dtt_schedule_empty, dtt_schedule_tile_chunks, dtt_schedule_whole, fill_desc,
               pointer_array)


def schedules_for(w) -> List[Schedule]:
    """Each rank's schedule for workload ``w`` from the library's builders."""
    out = []
    rb = w.row_bytes
    for r in range(w.P):
        if r not in w.senders():
            out.append(dtt_schedule_empty())
            continue
        off = w.slice_offset(r)
        if w.kind == "whole":
            out.append(dtt_schedule_whole(off, w.M, rb, rb, w.num_programs))
        elif w.kind == "chunks":
            out.append(dtt_schedule_chunks(off, w.M, rb, rb, w.num_chunks))
        elif w.kind == "tile_chunks":
            kind = ORDER_GROUPED if w.group_m else ORDER_ROW_MAJOR
            out.append(dtt_schedule_tile_chunks(off, w.M, w.N, w.elem_bytes, rb, w.BM, w.BN,
                                                w.tiles_per_chunk, kind, w.group_m))
        else:
            raise ValueError(f"unknown schedule kind {w.kind}")
    return out


def producer_steps(w) -> int:
    """Steps (tiles) of one rank's fill producer for workload ``w``."""
    if w.kind == "whole":
        BM = -(-w.M // w.num_programs)
        return -(-w.M // BM)
    if w.kind == "chunks":
        BM = -(-w.M // w.num_chunks)
        return -(-w.M // BM)
    return (-(-w.M // w.BM)) * (-(-w.N // w.BN))


def producer_desc(w, cluster: int = 1, programs: Optional[int] = None, threads: int = 0,
                  group: int = 1, counters=None, pace: int = 0):
    """The fill producer that matches ``w``'s schedule (same tiles, same order, same marks).
    group > 1: each program is `group` CTAs that mark each step once (counters: device int32
    [P * producer_steps(w)], zeroed).  pace > 0: a program waits for chunk k - pace of its rank
    to be delivered before it writes chunk k (timing only)."""
    slice_offs = [w.slice_offset(r) for r in range(w.P)]
    mask = 0
    for r in w.senders():
        mask |= 1 << r
    if w.kind == "whole":
        NP = w.num_programs
        BM = -(-w.M // NP)
        if group > 1:
            # each program is a group of CTAs that marks its one step once: the same NP marks as
            # one mark per program at the end, when every program has exactly one step
            if -(-w.M // BM) != NP:
                raise ValueError("group writers on whole() need one step per program")
            return fill_desc(w.dtype, w.seed, w.M, w.N, w.row_bytes, w.buf_bytes, slice_offs, BM, w.N, NP, NP,
                             mark_mode=MARK_PER_STEP, cluster=1, rank_mask=mask, threads=threads,
                             group=group, group_counters=counters, pace=pace)
        return fill_desc(w.dtype, w.seed, w.M, w.N, w.row_bytes, w.buf_bytes, slice_offs, BM, w.N, NP, 1,
                         mark_mode=MARK_AT_END, cluster=1, rank_mask=mask, threads=threads, pace=pace)
    if w.kind == "chunks":
        BM = -(-w.M // w.num_chunks)
        n = -(-w.M // BM)
        NP = programs or n
        return fill_desc(w.dtype, w.seed, w.M, w.N, w.row_bytes, w.buf_bytes, slice_offs, BM, w.N, NP, 1,
                         mark_mode=MARK_PER_STEP, cluster=cluster, rank_mask=mask, threads=threads,
                         group=group, group_counters=counters, pace=pace)
    kind = ORDER_GROUPED if w.group_m else ORDER_ROW_MAJOR
    return fill_desc(w.dtype, w.seed, w.M, w.N, w.row_bytes, w.buf_bytes, slice_offs, w.BM, w.BN,
                     programs or w.num_programs, w.tiles_per_chunk, order_kind=kind,
                     group_m=w.group_m, mark_mode=MARK_PER_STEP, cluster=cluster, rank_mask=mask,
                     threads=threads, group=group, group_counters=counters, pace=pace)


@dataclass
class Setup:
    w: object
    bufs: List[torch.Tensor]
    plan: Plan
    desc: object
    producer_stream: torch.cuda.Stream
    counters: Optional[torch.Tensor] = None
    buf_ptrs: object = None           # the buffers' addresses, marshalled once


def make(w, opts=None, cluster: int = 1, programs: Optional[int] = None, threads: int = 0,
         device: str = "cuda", fill_byte: int = 0, copy_stream=None, group: int = 1,
         pace: int = 0) -> Setup:
    """Allocate the P symmetric buffers (uint8, w.buf_bytes each), build the plan and producer.
    copy_stream: a non-blocking stream for the copier (None: the plan makes its own)."""
    bufs = [torch.full((w.buf_bytes,), fill_byte, dtype=torch.uint8, device=device)
            for _ in range(w.P)]
    scheds = schedules_for(w)
    if opts is None:
        opts = dtt_plan_opts_default()
    opts.allgather = 0 if w.broadcast else 1
    plan = Plan(bufs, w.buf_bytes, scheds, opts, copy_stream=copy_stream)
    for s in scheds:
        s.free()
    counters = None
    if group > 1:
        counters = torch.zeros(w.P * producer_steps(w), dtype=torch.int32, device=device)
    desc = producer_desc(w, cluster=cluster, programs=programs, threads=threads, group=group,
                         counters=counters, pace=pace)
    torch.cuda.synchronize()          # buffers initialised before any round starts
    return Setup(w, bufs, plan, desc, torch.cuda.Stream(), counters, pointer_array(bufs))


def run_round(st: Setup, raise_on_error: bool = True):
    """One round: start (launches the copier), the fill producer, wait.  Returns the report."""
    handles = st.plan.start(st.producer_stream)
    dtt_fill_producer(st.buf_ptrs, st.desc, handles, st.producer_stream)
    return st.plan.wait(raise_on_error=raise_on_error)


def run_overlapped(st: Setup, rounds: int, raise_on_error: bool = True, produce=None):
    """`rounds` rounds two at a time on a plan made with opts.overlap: round R is started and its
    producer launched before round R-1's wait (the producer waits, chunk by chunk, for round R-1's
    copies of what it overwrites), then the plan advances with round R still in flight.  The
    last round is waited for at the end.  produce(handles) launches a round's producer (default:
    the fill).  Returns the reports in round order."""
    reps = []
    for i in range(rounds):
        handles = st.plan.start(st.producer_stream)
        if produce is None:
            dtt_fill_producer(st.buf_ptrs, st.desc, handles, st.producer_stream)
        else:
            produce(handles)
        if st.plan.pending:
            reps.append(st.plan.wait(raise_on_error=raise_on_error))
        if i + 1 < rounds:
            st.plan.next_round()
    reps.append(st.plan.wait(raise_on_error=raise_on_error))
    return reps


def sm_count() -> int:
    """Streaming multiprocessors of the current CUDA device (the launch shapes below scale with
    it)."""
    return int(torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count)


def l2_bytes() -> int:
    """L2 size of the current CUDA device in bytes."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return int(getattr(props, "L2_cache_size", 0) or (129 << 20))


def bench_launch(w, overlap: Optional[bool] = None) -> dict:
    """The launch configuration the benchmark times for workload ``w`` (tests use it too).

    overlap: rounds two at a time (opts.overlap: a round's producer runs while the previous
    round's copier still copies).  None: where the benchmark uses them -- the chunked and GEMM
    workloads, and whole() with one step per program (c1, c4a).  The tiled fill's paced rounds
    already run at the DRAM roofline, and a round started early would only take its L2 away; a
    whole() slice written by many steps per program (the c4b broadcast) is one chunk, so its
    rounds have little to overlap, and its fill is fastest in 1024-thread CTAs, which cannot sit
    beside the copier's (overlapping rounds need that).

    Chunked workloads: the bulk-copy copier (six one-warp CTAs per SM, each with a ring of two
    16 KiB stages, so the producer keeps the SM's threads and registers), and one program per
    rank made of a group of SMs / P CTAs (one per SM in all) that writes the rank's chunks in
    order and marks each once, so every rank's chunk k opens in wave k and the copier follows the
    waves.  With overlapping rounds the producer is paced across rounds: it writes chunk k once
    chunk k - pace is delivered, chunk k < pace once the previous round's chunk n - pace + k is,
    with pace the number of chunk waves whose bytes fill about two thirds of L2, so the copier
    reads what the producer wrote from L2 and its next round's first chunks are ready when it
    starts (c2: ~106 -> ~92 us per round).  Rounds one at a time use the early copier instead:
    each round's copier launched by the previous round's wait and claimed by start (it waits up
    to 2 ms), so its launch leaves the round's critical path.
    whole(): the bulk-copy copier (two CTAs per SM, 2 x 56 KiB stages each) over the contiguous
    slices, launched after the producer's launch; the single chunk per rank opens only when the
    whole slice is written, so the fill gets as many CTAs as the writers allow.  A round of at
    most 2 MiB (c1) is latency-bound and gets the vector copier in 4 KiB pieces instead.
    tile_chunks (fill producer): the bulk-copy copier moving each 32 KiB tile as one tensor-map
    box (three CTAs per SM, two stages each), and a producer paced two chunks ahead of the
    copier (each program waits for chunk k - 2 of its rank to be delivered before it writes
    chunk k), so the copier reads what the producer wrote from L2; that needs every producer
    CTA resident at once (128-thread CTAs).  The GEMM producer keeps the vector copier: its own
    shared-memory ring leaves no room for a bulk-copy ring on the same SM."""
    sms = sm_count()
    if overlap is None:
        if w.kind == "whole":
            overlap = -(-w.M // -(-w.M // w.num_programs)) == w.num_programs
        else:
            overlap = w.kind == "chunks" or w.K > 0
    ov = 1 if overlap else 0
    early = 0 if overlap else 2000
    if w.kind == "chunks":     # six bulk-copy CTAs per SM: one thread alone cannot keep HBM busy
        launch = {"group": max(1, sms // len(w.senders())), "programs": 1, "threads": 256,
                  "opts": dtt_plan_opts_default(method=1, piece_bytes=16384, stages=2, ctas_per_sm=6,
                                                early_copier_us=early, overlap=ov)}
        if overlap:
            rows = -(-w.M // w.num_chunks)
            n = -(-w.M // rows)
            wave = len(w.senders()) * rows * w.row_bytes
            launch["pace"] = max(1, min(n, int(0.65 * l2_bytes() / wave)))
        return launch
    if w.kind == "whole":
        # the copier is launched after the producer's launch (it has nothing to do before the
        # whole slice is written)
        if len(w.senders()) * w.slice_bytes <= (2 << 20):
            # a round of at most 2 MiB is latency-bound: the vector copier in 4 KiB pieces spreads
            # each chunk over many CTAs (c1 gate-to-arrival 4.6 -> 3.4 us median)
            opts = dtt_plan_opts_default(method=0, piece_bytes=4096, copier_threads=256, ctas_per_sm=1,
                                         deferred_copier=2, overlap=ov)
        else:
            opts = dtt_plan_opts_default(method=1, piece_bytes=57344, stages=2, ctas_per_sm=2,
                                         deferred_copier=2, overlap=ov)
        NP = w.num_programs
        if -(-w.M // -(-w.M // NP)) == NP:
            # one step per program: each writer becomes a group of CTAs (up to 8, enough to
            # cover the SMs) that marks the chunk once
            g = max(1, min(8, sms // (len(w.senders()) * NP)))
            return {"group": g, "threads": 512, "opts": opts}
        # overlapping rounds: a producer CTA must fit on an SM beside the copier's
        return {"threads": 512 if overlap else 1024, "opts": opts}
    if w.K == 0:       # the tiled fill in 128-thread CTAs: all of them resident at once
        return {"threads": 128, "pace": 2,
                "opts": dtt_plan_opts_default(method=1, piece_bytes=32768, stages=2, ctas_per_sm=3,
                                              early_copier_us=early, overlap=ov)}
    # the GEMM producer: two 256-thread vector copier CTAs per SM beside the GEMM's CTA
    return {"opts": dtt_plan_opts_default(copier_threads=256, ctas_per_sm=2, early_copier_us=early,
                                          overlap=ov)}


@dataclass
class GemmSetup:
    w: object
    bufs: List[torch.Tensor]
    plan: Plan
    A: torch.Tensor
    Bt: torch.Tensor
    err: torch.Tensor
    producer_stream: torch.cuda.Stream
    num_programs: int
    buf_ptrs: object = None           # the buffers' addresses and slice offsets, marshalled once
    slice_offs: object = None


def make_gemm(w, A, Bt, opts=None, num_programs: Optional[int] = None, copy_stream=None) -> GemmSetup:
    """Plan + operands for the GEMM producer workload: each rank's slice is C_r, [M, N] bf16,
    tiled 128 x 128 and chunked by the producer's program count.  A [P, M, K] and Bt [N, K] are
    bf16 tensors (moved to the device here)."""
    from . import COPY_VEC16
    NP = num_programs or w.num_programs
    w = type(w)(**{**w.__dict__, "tiles_per_chunk": NP, "num_programs": NP})
    bufs = [torch.zeros(w.buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(w.P)]
    if opts is None:                  # the vector copier: it needs no shared memory
        opts = dtt_plan_opts_default(method=COPY_VEC16)
    opts.allgather = 1
    scheds = schedules_for(w)
    plan = Plan(bufs, w.buf_bytes, scheds, opts, copy_stream=copy_stream)
    for s in scheds:
        s.free()
    import ctypes
    offs = (ctypes.c_uint64 * w.P)(*[w.slice_offset(r) for r in range(w.P)])
    st = GemmSetup(w, bufs, plan, A.to("cuda").contiguous(), Bt.to("cuda").contiguous(),
                   torch.zeros(1, dtype=torch.int32, device="cuda"), torch.cuda.Stream(), NP,
                   pointer_array(bufs), offs)
    torch.cuda.synchronize()
    return st


def run_gemm_round(st: GemmSetup, raise_on_error: bool = True):
    from . import dtt_gemm_producer
    w = st.w
    handles = st.plan.start(st.producer_stream)
    dtt_gemm_producer(st.A, st.Bt, st.buf_ptrs, w.M, w.N, w.K, w.row_bytes, st.slice_offs,
                      st.num_programs, handles, st.err, st.producer_stream)
    return st.plan.wait(raise_on_error=raise_on_error)
