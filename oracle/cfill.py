"""Oracle: the producer's values from the plain-C restatement in ``oracle/fill.c``.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The same definition as ``oracle/hashfill.py`` (the build's own hash: the pages fix no value
formula), computed by scalar C loops so that full-size buffers can be compared byte for byte.
``fill.c`` is compiled with gcc into ``oracle/_fill.so`` on first use (or by ``build()``); rows
are split over host threads, each a ctypes call that releases the interpreter lock.
Pinned like ``hashfill`` (published MurmurHash3 vectors, torch's bf16 rounding, the uniform
closed form) and checked against ``hashfill`` element by element (tests/test_oracle_hash.py).
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "fill.c")
LIB = os.path.join(_HERE, "_fill.so")
DTYPES = {"bf16": (0, 2), "f32": (1, 4), "u8": (2, 1)}

_lib = None


def build() -> str:
    """Compile fill.c into _fill.so (plain gcc, no machine-specific flags)."""
    tmp = LIB + ".tmp"
    subprocess.run(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        L = C.CDLL(LIB)
        for name in ("oracle_fmix32", "oracle_uniform_bits", "oracle_bf16_bits"):
            getattr(L, name).restype = C.c_uint32
            getattr(L, name).argtypes = [C.c_uint32]
        L.oracle_salt.restype = C.c_uint32
        L.oracle_salt.argtypes = [C.c_uint32] * 3
        L.oracle_fill_rows.restype = C.c_int
        L.oracle_fill_rows.argtypes = [C.c_int, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64,
                                       C.c_uint64, C.c_uint64, C.c_void_p]
        _lib = L
    return _lib


def fmix32(h: int) -> int:
    return lib().oracle_fmix32(h & 0xFFFFFFFF)


def salt(seed: int, rank: int, rnd: int) -> int:
    return lib().oracle_salt(seed & 0xFFFFFFFF, rank & 0xFFFFFFFF, rnd & 0xFFFFFFFF)


def uniform_bits(h: int) -> int:
    return lib().oracle_uniform_bits(h & 0xFFFFFFFF)


def bf16_bits(f32_bits: int) -> int:
    return lib().oracle_bf16_bits(f32_bits & 0xFFFFFFFF)


def fill_rows_into(out: np.ndarray, dtype: str, seed: int, rank: int, rnd: int, N: int,
                   row0: int, row1: int, threads: int = 0) -> None:
    """Rows [row0, row1) of rank's slice for round rnd, as raw bytes, into the uint8 array
    ``out`` ((row1 - row0) * N * element bytes, contiguous)."""
    code, eb = DTYPES[dtype]
    row_bytes = N * eb
    assert out.dtype == np.uint8 and out.flags.c_contiguous
    assert out.nbytes == (row1 - row0) * row_bytes
    L = lib()
    base = out.ctypes.data
    n = row1 - row0
    threads = threads or min(32, os.cpu_count() or 1)
    per = max(1, -(-n // threads))

    def part(i):
        a = row0 + i * per
        b = min(row1, a + per)
        if a < b:
            rc = L.oracle_fill_rows(code, seed & 0xFFFFFFFF, rank, rnd & 0xFFFFFFFF, N, a, b,
                                    base + (a - row0) * row_bytes)
            assert rc == 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(part, range(-(-n // per))))


def fill_slice_bytes(dtype: str, seed: int, rank: int, rnd: int, M: int, N: int,
                     threads: int = 0) -> np.ndarray:
    """Rank's whole M x N slice for round rnd as raw little-endian bytes."""
    out = np.empty(M * N * DTYPES[dtype][1], dtype=np.uint8)
    fill_rows_into(out, dtype, seed, rank, rnd, N, 0, M, threads)
    return out


def expected_buffer(w, rnd: int, threads: int = 0) -> np.ndarray:
    """Closed form of every virtual rank's buffer after round rnd of workload ``w``
    ("Triggered Plans", section Model: each buffer ends up holding every rank's slice at its
    own offset; a broadcast's buffers all hold the sender's slice)."""
    out = np.empty(w.buf_bytes, dtype=np.uint8)
    S = w.slice_bytes
    for r in w.senders():
        off = w.slice_offset(r)
        fill_rows_into(out[off:off + S], w.dtype, w.seed, r, rnd, w.N, 0, w.M, threads)
    return out
