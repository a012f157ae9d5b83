"""Python binding of the triggered-plan library (libdtt.so, C ABI in include/dtt.h).

Argument marshalling only: every step of the path -- gate polls, copies, marks, checks,
barriers -- runs in the library's CUDA kernels.  PyTorch supplies device memory and streams;
buffers may be passed as torch tensors (their data pointer is used) or as integer device
addresses.  The functions keep the C names (``dtt_plan_create`` ...); ``Plan`` and ``Schedule``
are small owners around them.  Importing the package does not load the library; the first call
does, and raises if libdtt.so has not been built (build with
``python -m device_triggered_transfers_gb300.build``).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdtt.so")

MAX_RANKS = 16
REPORT_MAX = 64
GATE_WORDS = 8
(GATE_READY, GATE_ARRIVAL, GATE_COMPLETION, GATE_ERROR, GATE_COUNTER, GATE_T_OPEN,
 GATE_T_ARRIVE, GATE_COPIER) = range(8)

OK, EINVAL, EOUTOFROWS, EOVERLAP, ECAPACITY, EROUNDLIMIT, ESTATE, EEXTRA, ETIMEDOUT, ECUDA, \
    ENOMEM = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10
ERROR_NAMES = {OK: "OK", EINVAL: "EINVAL", EOUTOFROWS: "EOUTOFROWS", EOVERLAP: "EOVERLAP",
               ECAPACITY: "ECAPACITY", EROUNDLIMIT: "EROUNDLIMIT", ESTATE: "ESTATE",
               EEXTRA: "EEXTRA", ETIMEDOUT: "ETIMEDOUT", ECUDA: "ECUDA", ENOMEM: "ENOMEM"}
PREPARED, RUNNING, DONE, FAILED, CLOSING, CLOSED = range(6)
RC_CLOSING = 1      # dtt_plan_close left the plan CLOSING (not an error)
BF16, F32, U8 = 0, 1, 2
DTYPE_CODES = {"bf16": BF16, "f32": F32, "u8": U8}
ELEM_BYTES = {"bf16": 2, "f32": 4, "u8": 1}
COPY_VEC16, COPY_TMA, COPY_ENGINE = 0, 1, 2
ORDER_ROW_MAJOR, ORDER_GROUPED = 0, 1
MARK_PER_STEP, MARK_AT_END = 0, 1
HANDLE_TIMESTAMPS, HANDLE_OVERLAP = 1, 2
DEV_EBADCHUNK, DEV_EBADGROUP, DEV_EWRITABLE = 1, 2, 4


class dtt_region(C.Structure):
    _fields_ = [("offset", C.c_uint64), ("row_bytes", C.c_uint64), ("rows", C.c_uint64),
                ("pitch", C.c_uint64)]


class dtt_dest(C.Structure):
    _fields_ = [("offset", C.c_uint64), ("pitch", C.c_uint64)]


class dtt_order(C.Structure):
    _fields_ = [("kind", C.c_uint32), ("group_m", C.c_uint32)]


class dtt_plan_opts(C.Structure):
    _fields_ = [("allgather", C.c_uint32), ("method", C.c_uint32), ("copier_ctas", C.c_uint32),
                ("ctas_per_sm", C.c_uint32), ("copier_threads", C.c_uint32),
                ("piece_bytes", C.c_uint32), ("timestamps", C.c_uint32),
                ("initial_round", C.c_uint32), ("max_polls", C.c_uint64),
                ("max_regions", C.c_uint64), ("deferred_copier", C.c_uint32),
                ("stages", C.c_uint32), ("time_copier", C.c_uint32), ("host_piece_bytes", C.c_uint32),
                ("dst_bufs", C.c_void_p), ("dst_bytes", C.c_uint64), ("early_copier_us", C.c_uint32),
                ("overlap", C.c_uint32)]


class dtt_group_table(C.Structure):
    _fields_ = [("counters", C.c_void_p), ("size", C.c_void_p), ("chunk_off", C.c_void_p),
                ("chunk_ids", C.c_void_p), ("n_groups", C.c_uint32), ("reserved", C.c_uint32)]


class dtt_handle(C.Structure):
    _fields_ = [("gates", C.c_void_p), ("writers", C.c_void_p), ("status", C.c_void_p),
                ("round", C.c_uint32), ("rank", C.c_uint32), ("P", C.c_uint32),
                ("n_global", C.c_uint32), ("first_chunk", C.c_uint32), ("n_chunks", C.c_uint32),
                ("flags", C.c_uint32), ("reserved", C.c_uint32), ("groups", dtt_group_table),
                ("peer_masks", C.c_void_p), ("host_ready", C.c_void_p)]


class dtt_report(C.Structure):
    _fields_ = [("status", C.c_int32), ("n_short", C.c_uint32), ("n_extra", C.c_uint32),
                ("copier_timeouts", C.c_uint32), ("device_status", C.c_uint32),
                ("round", C.c_uint32), ("short_chunks", C.c_uint32 * REPORT_MAX),
                ("extra_chunks", C.c_uint32 * REPORT_MAX)]

    @property
    def shorts(self) -> List[int]:
        return list(self.short_chunks[:min(self.n_short, REPORT_MAX)])

    @property
    def extras(self) -> List[int]:
        return list(self.extra_chunks[:min(self.n_extra, REPORT_MAX)])


class dtt_fill_desc(C.Structure):
    _fields_ = [("dtype", C.c_uint32), ("seed", C.c_uint32), ("M", C.c_uint64),
                ("N", C.c_uint64), ("pitch", C.c_uint64), ("buf_bytes", C.c_uint64),
                ("slice_off", C.c_uint64 * MAX_RANKS),
                ("BM", C.c_uint32), ("BN", C.c_uint32), ("num_programs", C.c_uint32),
                ("tiles_per_chunk", C.c_uint32), ("order", dtt_order),
                ("mark_mode", C.c_uint32), ("cluster", C.c_uint32), ("rank_mask", C.c_uint32),
                ("threads", C.c_uint32), ("group", C.c_uint32), ("pace", C.c_uint32),
                ("group_counters", C.c_void_p)]


class dtt_allreduce_desc(C.Structure):
    _fields_ = [("dtype", C.c_uint32), ("sub_blocks", C.c_uint32), ("block_rows", C.c_uint64),
                ("cols", C.c_uint64), ("pitch", C.c_uint64), ("reduce_ctas", C.c_uint32),
                ("reduce_threads", C.c_uint32), ("scatter_only", C.c_uint32)]


ORDER_FN = C.CFUNCTYPE(C.c_int, C.c_uint64, C.c_void_p, C.POINTER(C.c_uint32),
                       C.POINTER(C.c_uint32))

_P = C.c_void_p
_u32, _u64, _i32 = C.c_uint32, C.c_uint64, C.c_int32
_SIGS = {
    "dtt_last_error": (C.c_char_p, []),
    "dtt_preload": (C.c_int, []),
    "dtt_tile_of": (C.c_int, [C.POINTER(dtt_order), _u64, _u32, _u32, C.POINTER(_u32), C.POINTER(_u32)]),
    "dtt_schedule_whole": (C.c_int, [_u64, _u64, _u64, _u64, _u32, C.POINTER(_P)]),
    "dtt_schedule_chunks": (C.c_int, [_u64, _u64, _u64, _u64, _u32, C.POINTER(_P)]),
    "dtt_schedule_tile_chunks": (C.c_int, [_u64, _u64, _u64, _u32, _u64, _u32, _u32, _u32,
                                           C.POINTER(dtt_order), ORDER_FN, _P, C.POINTER(_P)]),
    "dtt_schedule_empty": (C.c_int, [C.POINTER(_P)]),
    "dtt_schedule_add_chunk": (C.c_int, [_P, C.POINTER(dtt_region), _u32, _u32]),
    "dtt_schedule_add_chunk_to": (C.c_int, [_P, C.POINTER(dtt_region), C.POINTER(dtt_dest), _u32, _u32, _u32]),
    "dtt_schedule_get_dests": (C.c_int, [_P, _u32, C.POINTER(dtt_dest), _u64, C.POINTER(_u64), C.POINTER(_u32)]),
    "dtt_schedule_info": (C.c_int, [_P, C.POINTER(_u32), C.POINTER(_u64)]),
    "dtt_schedule_get": (C.c_int, [_P, _u32, C.POINTER(dtt_region), _u64, C.POINTER(_u64), C.POINTER(_u32)]),
    "dtt_schedule_free": (None, [_P]),
    "dtt_plan_opts_default": (None, [C.POINTER(dtt_plan_opts)]),
    "dtt_plan_create": (C.c_int, [C.POINTER(_P), _u64, _u32, C.POINTER(_P), C.POINTER(dtt_plan_opts),
                                  _P, C.POINTER(_P)]),
    "dtt_plan_start": (C.c_int, [_P, _P, C.POINTER(dtt_handle)]),
    "dtt_plan_handle": (C.c_int, [_P, _u32, C.POINTER(dtt_handle)]),
    "dtt_plan_launch_copier": (C.c_int, [_P]),
    "dtt_plan_wait": (C.c_int, [_P, C.POINTER(dtt_report)]),
    "dtt_plan_next_round": (C.c_int, [_P]),
    "dtt_plan_close": (C.c_int, [_P]),
    "dtt_plan_state": (C.c_int, [_P]),
    "dtt_plan_early_stats": (C.c_int, [_P, C.POINTER(_u64), C.POINTER(_u64), C.POINTER(_u64),
                                       C.POINTER(_u64)]),
    "dtt_plan_define_groups": (C.c_int, [_P, _u32, C.POINTER(_u32), C.POINTER(_u32)]),
    "dtt_plan_define_block_groups": (C.c_int, [_P, _u64, C.POINTER(_u32), C.POINTER(_u32)]),
    "dtt_plan_read_group_counters": (C.c_int, [_P, C.POINTER(_u64), _u64]),
    "dtt_plan_round": (C.c_uint32, [_P]),
    "dtt_plan_pending_round": (C.c_uint32, [_P]),
    "dtt_plan_info": (C.c_int, [_P, C.POINTER(_u32), C.POINTER(_u32), C.POINTER(_u32), C.POINTER(_P)]),
    "dtt_plan_read_gates": (C.c_int, [_P, C.POINTER(_u64), _u64]),
    "dtt_gemm_consumer": (C.c_int, [_P, C.c_uint32, _P, C.c_uint32, C.c_uint32, _P, _u64, C.c_uint32,
                                    _u64, _P, _P]),
    "dtt_plan_stats": (C.c_int, [_P, C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(_u64)]),
    "dtt_allgather_host": (C.c_int, [_P, C.POINTER(_P), _P, _u32, _P, C.POINTER(dtt_report)]),
    "dtt_allgather_host_rounds": (C.c_int, [_P, _u32, C.POINTER(_P), C.POINTER(_P), _u32, _P,
                                            C.POINTER(dtt_report)]),
    "dtt_fill_producer": (C.c_int, [C.POINTER(_P), _u32, C.POINTER(dtt_fill_desc),
                                    C.POINTER(dtt_handle), _P]),
    "dtt_publish": (C.c_int, [C.POINTER(dtt_handle), _u32, _u32, _u32, _u32, _P]),
    "dtt_gemm_producer": (C.c_int, [_P, _P, C.POINTER(_P), _u32, _u32, _u32, _u32, _u64,
                                    C.POINTER(_u64), _u32, C.POINTER(dtt_handle), _P, _P]),
    "dtt_consumer_gather": (C.c_int, [_P, _u32, _P, _u64, _P, _u32, _P]),
    "dtt_allreduce_create": (C.c_int, [C.POINTER(_P), _u64, C.POINTER(_P), _u64, _u32,
                                       C.POINTER(dtt_allreduce_desc), C.POINTER(dtt_plan_opts),
                                       C.POINTER(dtt_plan_opts), _P, _P, C.POINTER(_P)]),
    "dtt_allreduce_plans": (C.c_int, [_P, C.POINTER(_P), C.POINTER(_P)]),
    "dtt_allreduce_start": (C.c_int, [_P, _P, C.POINTER(dtt_handle)]),
    "dtt_allreduce_reduce": (C.c_int, [_P, _P, _P]),
    "dtt_allreduce_wait": (C.c_int, [_P, C.POINTER(dtt_report), C.POINTER(dtt_report)]),
    "dtt_allreduce_host": (C.c_int, [_P, C.POINTER(_P), _P, _u32, _P, _P, C.POINTER(dtt_report),
                                     C.POINTER(dtt_report)]),
    "dtt_allreduce_next_round": (C.c_int, [_P]),
    "dtt_allreduce_destroy": (C.c_int, [_P]),
    "dtt_barrier_handrolled": (C.c_int, [C.POINTER(_P), C.POINTER(_P), _u32, _u32, _u64, _P, _P]),
    "dtt_barrier_create": (C.c_int, [_u32, C.POINTER(_P)]),
    "dtt_barrier_destroy": (None, [_P]),
    "dtt_barrier_reveal": (C.c_int, [_P, C.POINTER(_P), C.POINTER(_P), C.POINTER(_P), _u32, _u64,
                                     _P, _P]),
    "dtt_barrier_reveal_noalloc": (C.c_int, [C.POINTER(_P), C.POINTER(_P), C.POINTER(_P), _u32,
                                             _u32, _u64, _P, _P]),
}

_lib = None


def lib():
    """The loaded libdtt.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libdtt.so not built at {LIB_PATH}; run "
                              "python -m device_triggered_transfers_gb300.build")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class DttError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _check(rc: int) -> int:
    if rc != OK:
        raise DttError(rc, lib().dtt_last_error().decode(errors="replace"))
    return rc


def _ptr(x) -> int:
    """Device (or host) address of a torch tensor, or an integer address."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _ptr_array(xs) -> C.Array:
    if isinstance(xs, C.Array):       # already marshalled (see pointer_array)
        return xs
    arr = (C.c_void_p * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x) or None
    return arr


def pointer_array(xs) -> C.Array:
    """The device addresses of ``xs`` (tensors or integers) as the C array the calls taking a
    buffer list expect; build it once and pass it instead of the list on every round."""
    return _ptr_array(list(xs))


# ---- schedules --------------------------------------------------------------------------------
class Schedule:
    """Owner of a dtt_schedule*."""

    def __init__(self, handle: int):
        self._h = C.c_void_p(handle)

    @property
    def handle(self) -> C.c_void_p:
        return self._h

    def info(self):
        n, r = _u32(), _u64()
        _check(lib().dtt_schedule_info(self._h, C.byref(n), C.byref(r)))
        return n.value, r.value

    @property
    def n_chunks(self) -> int:
        return self.info()[0]

    def chunk(self, i: int):
        """(list of (offset, row_bytes, rows, pitch), writers) of chunk i."""
        n, w = _u64(), _u32()
        _check(lib().dtt_schedule_get(self._h, i, None, 0, C.byref(n), C.byref(w)))
        regs = (dtt_region * max(1, n.value))()
        _check(lib().dtt_schedule_get(self._h, i, regs, n.value, C.byref(n), C.byref(w)))
        return [(r.offset, r.row_bytes, r.rows, r.pitch) for r in regs[:n.value]], w.value

    def chunks(self):
        return [self.chunk(i) for i in range(self.n_chunks)]

    def add_chunk(self, regions, writers: int, dests=None, peers: int = 0) -> None:
        """regions: (offset, row_bytes, rows, pitch) tuples; dests (optional): one (offset, pitch)
        per region, where it lands; peers: bit mask of receiving ranks (0: every other rank)."""
        arr = (dtt_region * max(1, len(regions)))(*[dtt_region(*r) for r in regions])
        if dests is None and not peers:
            _check(lib().dtt_schedule_add_chunk(self._h, arr, len(regions), writers))
            return
        d = None
        if dests is not None:
            if len(dests) != len(regions):
                raise DttError(EINVAL, "add_chunk: one destination per region")
            d = (dtt_dest * max(1, len(dests)))(*[dtt_dest(*x) for x in dests])
        _check(lib().dtt_schedule_add_chunk_to(self._h, arr, d, len(regions), writers, peers))

    def dests(self, i: int):
        """(list of (offset, pitch) or None when chunk i lands at its own offsets, peer mask)."""
        n, m = _u64(), _u32()
        _check(lib().dtt_schedule_get_dests(self._h, i, None, 0, C.byref(n), C.byref(m)))
        if n.value == 0:
            return None, m.value
        arr = (dtt_dest * n.value)()
        _check(lib().dtt_schedule_get_dests(self._h, i, arr, n.value, C.byref(n), C.byref(m)))
        return [(x.offset, x.pitch) for x in arr], m.value

    def free(self) -> None:
        if self._h and self._h.value:
            lib().dtt_schedule_free(self._h)
            self._h = C.c_void_p(0)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def dtt_schedule_whole(base_off, rows, row_bytes, pitch, num_programs) -> Schedule:
    out = C.c_void_p()
    _check(lib().dtt_schedule_whole(base_off, rows, row_bytes, pitch, num_programs, C.byref(out)))
    return Schedule(out.value)


def dtt_schedule_chunks(base_off, rows, row_bytes, pitch, num_chunks) -> Schedule:
    out = C.c_void_p()
    _check(lib().dtt_schedule_chunks(base_off, rows, row_bytes, pitch, num_chunks, C.byref(out)))
    return Schedule(out.value)


def dtt_schedule_tile_chunks(base_off, M, N, elem_bytes, pitch, BM, BN, tiles_per_chunk,
                             order_kind=ORDER_ROW_MAJOR, group_m=0, order_fn=None) -> Schedule:
    """order_fn: optional Python callable step -> (tm, tn) (host-side mapping)."""
    out = C.c_void_p()
    order = dtt_order(order_kind, group_m)
    if order_fn is not None:
        def cb(step, ctx, tm, tn):
            try:
                a, b = order_fn(step)
                tm[0], tn[0] = a, b
                return 0
            except Exception:
                return 1
        fn = ORDER_FN(cb)
    else:
        fn = ORDER_FN()
    _check(lib().dtt_schedule_tile_chunks(base_off, M, N, elem_bytes, pitch, BM, BN, tiles_per_chunk,
                                          C.byref(order), fn, None, C.byref(out)))
    return Schedule(out.value)


def dtt_schedule_empty() -> Schedule:
    out = C.c_void_p()
    _check(lib().dtt_schedule_empty(C.byref(out)))
    return Schedule(out.value)


# ---- schedules from tensor slices, in the pages' form ---------------------------------------------
# "Triggered Plans" (section Model) builds a rank's schedule from its own part of the output,
# `mine`, a view into the output tensor `base`: whole(mine), chunks(mine, n, base=out) and
# tile_chunks(mine, (BM, BN), tiles_per_chunk, order=..., base=out).  The functions below take
# the same arguments (torch tensors) and turn them into the byte offset, row bytes and pitch of
# the C builders; regions are relative to base's first byte.

def _slice_geometry(mine, base):
    """(offset of mine's first byte in base, rows, row bytes, pitch in bytes, element bytes, cols)
    of a 1D or 2D view `mine` whose rows are contiguous."""
    e = mine.element_size()
    if mine.dim() == 1:
        rows, cols, pitch = 1, mine.shape[0], mine.shape[0] * e
        if mine.shape[0] and mine.stride(0) != 1:
            raise DttError(EINVAL, "schedule: a 1D slice must be contiguous")
    elif mine.dim() == 2:
        rows, cols = mine.shape
        if cols > 1 and mine.stride(1) != 1:
            raise DttError(EINVAL, "schedule: a slice's rows must be contiguous")
        pitch = mine.stride(0) * e if rows > 1 else cols * e
    else:
        raise DttError(EINVAL, "schedule: the slice must be 1D or 2D")
    off = 0
    if base is not None:
        off = mine.data_ptr() - base.data_ptr()
        if off < 0 or off + max(0, rows - 1) * pitch + cols * e > base.numel() * base.element_size():
            raise DttError(EINVAL, "schedule: the slice lies outside base")
    return off, rows, cols * e, pitch, e, cols


def whole(mine, num_programs: int = 1, base=None) -> Schedule:
    """One chunk holding all of `mine`, marked once by each of num_programs programs at their end."""
    off, rows, rb, pitch, _, _ = _slice_geometry(mine, base)
    return dtt_schedule_whole(off, rows, rb, pitch, num_programs)


def chunks(mine, n: int, base=None) -> Schedule:
    """Row blocks of `mine` completed in order, one writer each."""
    off, rows, rb, pitch, _, _ = _slice_geometry(mine, base)
    return dtt_schedule_chunks(off, rows, rb, pitch, n)


def tile_chunks(mine, tile, tiles_per_chunk: int, order=None, base=None) -> Schedule:
    """Consecutive (BM, BN) tiles of a tiled producer over `mine`, tiles_per_chunk steps per chunk.
    order: None (row-major), ("grouped", GROUP_M) (the library's grouped order), or a callable
    step -> (tm, tn), the producer's own mapping."""
    off, rows, _, pitch, e, cols = _slice_geometry(mine, base)
    BM, BN = tile
    if order is None:
        return dtt_schedule_tile_chunks(off, rows, cols, e, pitch, BM, BN, tiles_per_chunk)
    if isinstance(order, tuple) and len(order) == 2 and order[0] == "grouped":
        return dtt_schedule_tile_chunks(off, rows, cols, e, pitch, BM, BN, tiles_per_chunk,
                                        ORDER_GROUPED, int(order[1]))
    if callable(order):
        return dtt_schedule_tile_chunks(off, rows, cols, e, pitch, BM, BN, tiles_per_chunk, order_fn=order)
    raise DttError(EINVAL, "tile_chunks: order is None, ('grouped', GROUP_M) or a callable")


def dtt_tile_of(order_kind, group_m, step, tiles_m, tiles_n):
    tm, tn = _u32(), _u32()
    order = dtt_order(order_kind, group_m)
    _check(lib().dtt_tile_of(C.byref(order), step, tiles_m, tiles_n, C.byref(tm), C.byref(tn)))
    return tm.value, tn.value


# ---- plans ------------------------------------------------------------------------------------
def dtt_plan_opts_default(**over) -> dtt_plan_opts:
    o = dtt_plan_opts()
    lib().dtt_plan_opts_default(C.byref(o))
    for k, v in over.items():
        setattr(o, k, v)
    return o


class Plan:
    """Owner of a dtt_plan* over P device buffers (kept alive here)."""

    def __init__(self, bufs: Sequence, buf_bytes: int, schedules: Sequence[Optional[Schedule]],
                 opts: Optional[dtt_plan_opts] = None, copy_stream=None, dst_bufs=None,
                 dst_bytes: int = 0):
        """dst_bufs (optional): P separate destination buffers of dst_bytes each that every copy
        lands in (opts.dst_bufs)."""
        self.bufs = list(bufs)
        self.P = len(self.bufs)
        self.buf_bytes = buf_bytes
        self.copy_stream = copy_stream
        self.dst_bufs = list(dst_bufs) if dst_bufs is not None else None
        if dst_bufs is not None:
            if len(self.dst_bufs) != self.P:
                raise DttError(EINVAL, "Plan: one destination buffer per rank")
            opts = dtt_plan_opts.from_buffer_copy(opts) if opts is not None else dtt_plan_opts_default()
            self._dst_arr = _ptr_array(self.dst_bufs)
            opts.dst_bufs = C.cast(self._dst_arr, C.c_void_p).value
            opts.dst_bytes = dst_bytes
        scheds = (C.c_void_p * self.P)(*[(s.handle.value if s is not None else None)
                                         for s in schedules])
        out = C.c_void_p()
        _check(lib().dtt_plan_create(_ptr_array(self.bufs), buf_bytes, self.P, scheds,
                                     C.byref(opts) if opts is not None else None,
                                     _stream(copy_stream), C.byref(out)))
        self._h = out
        self.handles = (dtt_handle * self.P)()
        # the round's calls, looked up once (a round is four calls; their lookups are not free)
        L = lib()
        self._start, self._wait, self._next = L.dtt_plan_start, L.dtt_plan_wait, L.dtt_plan_next_round
        self._stream_obj, self._stream_int = None, 0

    # the round
    def start(self, producer_stream=None):
        if producer_stream is not self._stream_obj:
            self._stream_obj, self._stream_int = producer_stream, _stream(producer_stream)
        rc = self._start(self._h, self._stream_int, self.handles)
        if rc:
            _check(rc)
        return self.handles

    def launch_copier(self) -> None:
        _check(lib().dtt_plan_launch_copier(self._h))

    def handle(self, rank: int) -> dtt_handle:
        h = dtt_handle()
        _check(lib().dtt_plan_handle(self._h, rank, C.byref(h)))
        return h

    def wait(self, raise_on_error: bool = True) -> dtt_report:
        rep = dtt_report()
        rc = self._wait(self._h, C.byref(rep))
        if rc and raise_on_error:
            _check(rc)
        return rep

    def next_round(self) -> int:
        rc = self._next(self._h)
        if rc:
            _check(rc)
        return self.round

    def close(self) -> int:
        """Close the plan.  Returns OK, or RC_CLOSING when its copier waits behind an earlier
        plan's copier on the same copy stream: the plan is then CLOSING, closing the earlier
        plan finishes it, and a second close() releases it."""
        if self._h and self._h.value:
            rc = lib().dtt_plan_close(self._h)
            if rc == RC_CLOSING:
                return rc
            self._h = C.c_void_p(0)
            _check(rc)
        return OK

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def state(self) -> int:
        if not (self._h and self._h.value):
            return CLOSED
        return lib().dtt_plan_state(self._h)

    @property
    def round(self) -> int:
        return lib().dtt_plan_round(self._h)

    @property
    def pending(self) -> int:
        """The round in flight behind the current one (opts.overlap), or 0."""
        return lib().dtt_plan_pending_round(self._h)

    def info(self):
        n = _u32()
        first = (C.c_uint32 * self.P)()
        cnt = (C.c_uint32 * self.P)()
        gates = C.c_void_p()
        _check(lib().dtt_plan_info(self._h, C.byref(n), first, cnt, C.byref(gates)))
        return n.value, list(first), list(cnt), gates.value

    def stats(self):
        """(copier_ms_last, copier_ms_total, rounds_timed) for plans with opts.time_copier."""
        last, total, n = C.c_double(), C.c_double(), _u64()
        _check(lib().dtt_plan_stats(self._h, C.byref(last), C.byref(total), C.byref(n)))
        return last.value, total.value, n.value

    def define_groups(self, groups) -> int:
        """Chunk groups (lists of global chunk ids), before the first start; see
        dtt_plan_define_groups.  Returns the number of groups."""
        groups = [list(g) for g in groups]
        offs = [0]
        for g in groups:
            offs.append(offs[-1] + len(g))
        o = (_u32 * len(offs))(*offs)
        ids = (_u32 * max(1, offs[-1]))(*[c for g in groups for c in g])
        _check(lib().dtt_plan_define_groups(self._h, len(groups), o, ids))
        self.n_groups = len(groups)
        return self.n_groups

    def define_block_groups(self, block_bytes: int):
        """One group per block of block_bytes bytes (the chunks touching it); returns
        (n_groups, [group id of each block or None])."""
        nb = -(-self.buf_bytes // block_bytes)
        n = _u32()
        bg = (_u32 * nb)()
        _check(lib().dtt_plan_define_block_groups(self._h, block_bytes, C.byref(n), bg))
        self.n_groups = n.value
        return n.value, [None if x == 0xFFFFFFFF else x for x in bg]

    def read_group_counters(self) -> np.ndarray:
        """The group counters as a uint64 array [P, n_groups]."""
        out = np.zeros((self.P, self.n_groups), dtype=np.uint64)
        _check(lib().dtt_plan_read_group_counters(self._h, out.ctypes.data_as(C.POINTER(_u64)), out.size))
        return out

    def early_stats(self) -> dict:
        """Early copiers so far (opts.early_copier_us): launched, claimed, expired, aborted."""
        v = [_u64() for _ in range(4)]
        _check(lib().dtt_plan_early_stats(self._h, *[C.byref(x) for x in v]))
        return dict(zip(("launched", "claimed", "expired", "aborted"), (x.value for x in v)))

    def read_gates(self) -> np.ndarray:
        """The P gate tables as a uint64 array [P, n_global, 8]."""
        n = self.info()[0]
        out = np.zeros((self.P, n, GATE_WORDS), dtype=np.uint64)
        _check(lib().dtt_plan_read_gates(self._h, out.ctypes.data_as(C.POINTER(_u64)), out.size))
        return out

    def allgather_host(self, host_slices: Sequence, host_out=None, out_rank: int = 0,
                       stream=None, raise_on_error: bool = True) -> dtt_report:
        rep = dtt_report()
        rc = lib().dtt_allgather_host(self._h, _ptr_array(host_slices), _ptr(host_out) or None,
                                      out_rank, _stream(stream), C.byref(rep))
        if raise_on_error:
            _check(rc)
        return rep

    def allgather_host_rounds(self, host_slices: Sequence[Sequence], host_outs=None, out_rank: int = 0,
                              stream=None, raise_on_error: bool = True) -> List[dtt_report]:
        """Several host-buffer rounds back to back, pipelined (dtt_allgather_host_rounds).
        host_slices: one list of P slices per round (None: as it stands); host_outs: one buffer
        (or None) per round, or None.  Returns the rounds' reports."""
        n = len(host_slices)
        if any(len(sl) != self.P for sl in host_slices):
            raise DttError(EINVAL, "allgather_host_rounds: P slices per round")
        if host_outs is not None and len(host_outs) != n:
            raise DttError(EINVAL, "allgather_host_rounds: one output (or None) per round")
        slices = _ptr_array([x for sl in host_slices for x in sl])
        outs = _ptr_array(list(host_outs)) if host_outs is not None else None
        reps = (dtt_report * max(1, n))()
        rc = lib().dtt_allgather_host_rounds(self._h, n, slices, outs, out_rank, _stream(stream), reps)
        if raise_on_error:
            _check(rc)
        return list(reps[:n])

    def gemm_consumer(self, rank: int, Wt, D, N: int, K: int, err, ldd: int = 0,
                      num_programs: int = 0, max_polls: int = 0, stream=None) -> None:
        """D = X . W^T over rank `rank`'s gathered buffer, each row block loaded once its chunks
        have arrived (see dtt_gemm_consumer)."""
        _check(lib().dtt_gemm_consumer(self._h, rank, _ptr(Wt), N, K, _ptr(D), ldd or 2 * N,
                                       num_programs, max_polls, _ptr(err), _stream(stream)))

    def consumer_gather(self, rank: int, dst, max_polls: int, status, ctas: int, stream) -> None:
        _check(lib().dtt_consumer_gather(self._h, rank, _ptr(dst), max_polls, _ptr(status), ctas,
                                         _stream(stream)))


def dtt_plan_create(bufs, buf_bytes, schedules, opts=None, copy_stream=None) -> Plan:
    return Plan(bufs, buf_bytes, schedules, opts, copy_stream)


class TriggeredPlan(Plan):
    """The pages' TriggeredPlan(ctx, out, schedules) for P virtual ranks: `outs` is the list of
    the P ranks' output tensors (one size), `schedules` one schedule per rank built from slices of
    them (whole / chunks / tile_chunks with base=outs[r]).  free_schedules: free the schedules once
    the plan has taken its own copy (the default)."""

    def __init__(self, outs: Sequence, schedules: Sequence[Optional[Schedule]], opts=None,
                 copy_stream=None, allgather: bool = False, free_schedules: bool = True):
        nbytes = [t.numel() * t.element_size() for t in outs]
        if len(set(nbytes)) != 1:
            raise DttError(EINVAL, "TriggeredPlan: the P outputs have one size")
        opts = dtt_plan_opts.from_buffer_copy(opts) if opts is not None else dtt_plan_opts_default()
        opts.allgather = 1 if allgather else 0
        super().__init__(list(outs), nbytes[0], schedules, opts, copy_stream=copy_stream)
        self.outs = list(outs)
        if free_schedules:
            for sc in schedules:
                if sc is not None:
                    sc.free()


def prepare_all_gather(outs: Sequence, schedules: Optional[Sequence[Optional[Schedule]]] = None, opts=None,
                       copy_stream=None) -> TriggeredPlan:
    """The pages' ctx.ccl.prepare_all_gather(out, schedule) for P virtual ranks: an in-place
    all-gather plan over the P outputs whose rank r owns rows [r*M, (r+1)*M) of its output (M =
    rows / P, the outputs seen as 2D [rows, ...] tensors), checking that each schedule stays inside
    its rank's rows.  schedules None: whole() of each rank's rows, as on the pages."""
    P = len(outs)
    if schedules is None:
        schedules = []
        for r, out in enumerate(outs):
            o2 = out if out.dim() == 2 else out.reshape(out.shape[0], -1)
            M = o2.shape[0] // P
            schedules.append(whole(o2[r * M:(r + 1) * M], 1, base=out))
    return TriggeredPlan(outs, schedules, opts, copy_stream, allgather=True)


# ---- two-shot all-reduce --------------------------------------------------------------------
class PlanView(Plan):
    """A plan owned by something else (an all-reduce's two plans): the read calls of Plan
    (info, read_gates, read_group_counters, stats), never closed from here."""

    def __init__(self, handle: C.c_void_p, bufs: Sequence, buf_bytes: int, n_groups: int = 0):
        self._h = handle
        self.bufs = list(bufs)
        self.P = len(self.bufs)
        self.buf_bytes = buf_bytes
        self.n_groups = n_groups

    def close(self) -> int:
        return OK

    def __del__(self):
        pass


class AllReduce:
    """Owner of a dtt_allreduce*: the two-shot all-reduce over P device buffers (see
    dtt_allreduce_create).  Rank r's vector is P * block_rows rows of `cols` elements of `dtype`
    at the start of bufs[r]; every rank ends with the sum of the P vectors there (gather=False:
    a reduce-scatter, rank b ends with the sum over its own block b only).  A round: start() ->
    handles for the producers' reduce-scatter marks, the producers, reduce(), wait(),
    next_round()."""

    def __init__(self, bufs: Sequence, buf_bytes: int, dtype: str, block_rows: int, cols: int,
                 sub_blocks: int = 1, pitch: int = 0, staging: Optional[Sequence] = None,
                 staging_bytes: int = 0, rs_opts: Optional[dtt_plan_opts] = None,
                 ag_opts: Optional[dtt_plan_opts] = None, reduce_ctas: int = 0, reduce_threads: int = 0,
                 rs_copy_stream=None, ag_copy_stream=None, gather: bool = True):
        self.bufs = list(bufs)
        self.P = len(self.bufs)
        self.staging = list(staging) if staging is not None else None
        if self.staging is not None and len(self.staging) != self.P:
            raise DttError(EINVAL, "AllReduce: one staging buffer per rank")
        self.buf_bytes, self.dtype = buf_bytes, dtype
        self.block_rows, self.cols, self.sub_blocks = block_rows, cols, sub_blocks
        d = dtt_allreduce_desc()
        d.dtype = DTYPE_CODES[dtype]
        d.sub_blocks, d.block_rows, d.cols, d.pitch = sub_blocks, block_rows, cols, pitch
        d.reduce_ctas, d.reduce_threads = reduce_ctas, reduce_threads
        d.scatter_only = 0 if gather else 1
        self.gather = gather
        self.desc = d
        out = C.c_void_p()
        stg = _ptr_array(self.staging) if self.staging is not None else None
        _check(lib().dtt_allreduce_create(_ptr_array(self.bufs), buf_bytes, stg, staging_bytes, self.P,
                                          C.byref(d), C.byref(rs_opts) if rs_opts is not None else None,
                                          C.byref(ag_opts) if ag_opts is not None else None,
                                          _stream(rs_copy_stream), _stream(ag_copy_stream), C.byref(out)))
        self._h = out
        self.handles = (dtt_handle * self.P)()
        rs, ag = C.c_void_p(), C.c_void_p()
        _check(lib().dtt_allreduce_plans(self._h, C.byref(rs), C.byref(ag)))
        self.rs = PlanView(rs, self.bufs, buf_bytes, n_groups=self.P * sub_blocks)
        self.ag = PlanView(ag, self.bufs, buf_bytes) if gather else None

    def start(self, producer_stream=None):
        _check(lib().dtt_allreduce_start(self._h, _stream(producer_stream), self.handles))
        return self.handles

    def reduce(self, err, stream=None) -> None:
        _check(lib().dtt_allreduce_reduce(self._h, _ptr(err), _stream(stream)))

    def wait(self, raise_on_error: bool = True):
        a, b = dtt_report(), dtt_report()
        rc = lib().dtt_allreduce_wait(self._h, C.byref(a), C.byref(b))
        if rc and raise_on_error:
            _check(rc)
        return a, b

    def host_round(self, host_parts: Sequence, err, host_out=None, out_rank: int = 0, stream=None,
                   raise_on_error: bool = True):
        """One round from host memory (dtt_allreduce_host): host_parts, P pinned host tensors
        (None: that rank's vector as it stands), each rank's vector with its rows back to back;
        host_out (pinned, or None) receives out_rank's result.  Returns both reports."""
        if len(host_parts) != self.P:
            raise DttError(EINVAL, "host_round: one host vector (or None) per rank")
        need = self.P * self.block_rows * self.cols * ELEM_BYTES[self.dtype]
        for i, x in enumerate(list(host_parts) + [host_out]):
            if x is None:
                continue
            if x.device.type != "cpu" or x.numel() * x.element_size() < need:
                raise DttError(EINVAL, f"host_round: host buffer {i} must be host memory of at least {need} bytes")
        a, b = dtt_report(), dtt_report()
        rc = lib().dtt_allreduce_host(self._h, _ptr_array(host_parts), _ptr(host_out) or None, out_rank,
                                      _ptr(err), _stream(stream), C.byref(a), C.byref(b))
        if rc and raise_on_error:
            _check(rc)
        return a, b

    def next_round(self) -> None:
        _check(lib().dtt_allreduce_next_round(self._h))

    def close(self) -> int:
        if self._h and self._h.value:
            rc = lib().dtt_allreduce_destroy(self._h)
            self._h = C.c_void_p(0)
            _check(rc)
        return OK

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- producers and barriers -----------------------------------------------------------------
def fill_desc(dtype: str, seed: int, M: int, N: int, pitch: int, buf_bytes: int,
              slice_offs: Sequence[int], BM: int, BN: int, num_programs: int, tiles_per_chunk: int,
              order_kind=ORDER_ROW_MAJOR, group_m=0, mark_mode=MARK_PER_STEP, cluster=1,
              rank_mask=None, threads=0, group=1, group_counters=None, pace=0) -> dtt_fill_desc:
    d = dtt_fill_desc()
    d.group = group
    d.pace = pace
    d.group_counters = _ptr(group_counters) or None
    d.dtype = DTYPE_CODES[dtype]
    d.seed = seed & 0xFFFFFFFF
    d.M, d.N, d.pitch, d.buf_bytes = M, N, pitch, buf_bytes
    for i, o in enumerate(slice_offs):
        d.slice_off[i] = o
    d.BM, d.BN, d.num_programs, d.tiles_per_chunk = BM, BN, num_programs, tiles_per_chunk
    d.order = dtt_order(order_kind, group_m)
    d.mark_mode, d.cluster = mark_mode, cluster
    d.rank_mask = ((1 << len(slice_offs)) - 1) if rank_mask is None else rank_mask
    d.threads = threads
    return d


def dtt_fill_producer(bufs, desc: dtt_fill_desc, handles, stream=None) -> None:
    rc = lib().dtt_fill_producer(_ptr_array(bufs), len(bufs), C.byref(desc), handles, _stream(stream))
    if rc:
        _check(rc)


def dtt_publish(handles, first_chunk: int, n_chunks: int, marks: int = 0, stream=None) -> None:
    _check(lib().dtt_publish(handles, len(handles), first_chunk, n_chunks, marks, _stream(stream)))


class HandrolledArgs:
    """The hand-rolled barrier's windows checked once and marshalled (see RevealArgs)."""

    def __init__(self, signal, y, status):
        P = len(signal)
        _check_handrolled_args(P, signal, y, status)
        self.P = P
        self.signal, self.y, self.status = _ptr_array(signal), _ptr_array(y), _ptr(status)
        self._keep = (signal, y, status)


def dtt_barrier_handrolled(signal, y=None, gen: int = 1, max_polls: int = 1 << 24, status=None,
                           stream=None) -> None:
    """signal may be a HandrolledArgs (then y and status come from it)."""
    a = signal if isinstance(signal, HandrolledArgs) else HandrolledArgs(signal, y, status)
    rc = lib().dtt_barrier_handrolled(a.signal, a.y, a.P, gen, max_polls, a.status, _stream(stream))
    if rc:
        _check(rc)


def _check_handrolled_args(P, signal, y, status) -> None:
    if len(y) != P:
        raise DttError(EINVAL, f"dtt_barrier_handrolled: y has {len(y)} windows, need P = {P}")
    for name, lst in (("signal", signal), ("y", y)):
        for r, t in enumerate(lst):
            n = _elements(t)
            if t is None or (n is not None and n < P):
                raise DttError(EINVAL, f"dtt_barrier_handrolled: {name}[{r}] holds {n} int32, need P = {P}")
    n = _elements(status)
    if status is None or (n is not None and n < P):
        raise DttError(EINVAL, f"dtt_barrier_handrolled: status holds {n} int32, need P = {P}")


def _elements(t) -> Optional[int]:
    """Element count of a tensor argument; None for a raw address (its size is unknown here)."""
    if t is None or isinstance(t, int):
        return None
    return int(t.numel())


def _check_reveal_args(who: str, P: int, x, data, y, size: int, status) -> None:
    """The reveal reads x[r] and writes data[r] and y[r] (size int32 each) for every rank r < P,
    and status[r]: refuse short lists and short tensors before the kernel could run past them."""
    if isinstance(x, C.Array) or isinstance(data, C.Array) or isinstance(y, C.Array):
        raise DttError(EINVAL, f"{who}: pass lists of P slices, not marshalled arrays")
    for name, lst in (("x", x), ("data", data), ("y", y)):
        if len(lst) != P:
            raise DttError(EINVAL, f"{who}: {name} has {len(lst)} slices, need P = {P}")
        for r, t in enumerate(lst):
            n = _elements(t)
            if t is None or (n is not None and n < size):
                raise DttError(EINVAL, f"{who}: {name}[{r}] holds {n} int32, need size = {size}")
            if n is not None and getattr(t, "element_size", lambda: 4)() != 4:
                raise DttError(EINVAL, f"{who}: {name}[{r}] is not a 4-byte (int32) tensor")
    n = _elements(status)
    if status is None or (n is not None and n < P):
        raise DttError(EINVAL, f"{who}: status holds {n} int32, need P = {P}")


class RevealArgs:
    """The reveal's slices checked once (lengths, sizes, element type) and marshalled: pass it to
    Barrier.reveal / dtt_barrier_reveal_noalloc in place of the three lists and the status
    tensor when the same buffers are used call after call."""

    def __init__(self, x, data, y, size: int, status, P: Optional[int] = None, who="reveal"):
        P = len(x) if P is None else P
        _check_reveal_args(who, P, x, data, y, size, status)
        self.P, self.size = P, size
        self.x, self.data, self.y = _ptr_array(x), _ptr_array(data), _ptr_array(y)
        self.status = _ptr(status)
        self._keep = (x, data, y, status)      # the tensors stay alive with the arrays


class Barrier:
    """Owner of the builtin barrier's state (dtt_barrier*)."""

    def __init__(self, P: int):
        out = C.c_void_p()
        _check(lib().dtt_barrier_create(P, C.byref(out)))
        self._h = out
        self.P = P

    def reveal(self, x, data=None, y=None, size: int = 0, max_polls: int = 1 << 24, status=None,
               stream=None) -> None:
        """y[r] = data[(r + 1) % P] after each rank staged x[r] into data[r] (see
        dtt_barrier_reveal).  x may be a RevealArgs (then data, y, size and status come from it)."""
        a = x if isinstance(x, RevealArgs) else RevealArgs(x, data, y, size, status, self.P, "Barrier.reveal")
        if a.P != self.P:
            raise DttError(EINVAL, f"Barrier.reveal: arguments for {a.P} ranks, barrier of {self.P}")
        rc = lib().dtt_barrier_reveal(self._h, a.x, a.data, a.y, a.size, max_polls, a.status, _stream(stream))
        if rc:
            _check(rc)

    def destroy(self) -> None:
        if self._h and self._h.value:
            lib().dtt_barrier_destroy(self._h)
            self._h = C.c_void_p(0)

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def dtt_barrier_create(P: int) -> Barrier:
    return Barrier(P)


def dtt_barrier_reveal_noalloc(x, data=None, y=None, size: int = 0, max_polls: int = 1 << 24,
                               status=None, stream=None) -> None:
    """The builtin reveal with its counters in the library's fixed device array: allocates
    nothing (for callers that cannot allocate device memory at call time).  Calls that overlap
    on the GPU share that array and race; run them on one stream.  x may be a RevealArgs."""
    a = x if isinstance(x, RevealArgs) else RevealArgs(x, data, y, size, status, None,
                                                       "dtt_barrier_reveal_noalloc")
    _check(lib().dtt_barrier_reveal_noalloc(a.x, a.data, a.y, a.P, a.size, max_polls, a.status,
                                            _stream(stream)))


def dtt_gemm_producer(A, Bt, bufs, M: int, N: int, K: int, ldc: int, slice_offs, num_programs: int,
                      handles, err, stream=None) -> None:
    """C_r = A_r . B for every rank (tcgen05 GEMM), marking each tile's chunk; see dtt.h."""
    offs = slice_offs if isinstance(slice_offs, C.Array) else (C.c_uint64 * len(bufs))(*slice_offs)
    _check(lib().dtt_gemm_producer(_ptr(A), _ptr(Bt), _ptr_array(bufs), len(bufs), M, N, K, ldc, offs,
                                   num_programs, handles, _ptr(err), _stream(stream)))
