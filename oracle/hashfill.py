"""Oracle: the producer's synthetic values, hash(seed, rank, round, row, col) -> [-1, 1).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The Iris "Triggered Plans" page (section Model) has its producer "compute and store the tile"
without saying what it stores; the workloads here store hashed values so that every element
depends on the round (the stale-data check that "Triggered SDMA Plans", section Testing,
describes: 8 writers on one gate over 10 rounds).  The formula is therefore this build's own
definition, not the pages':

* ``fmix32`` is the 32-bit finaliser of MurmurHash3 (Austin Appleby's public-domain hash),
  written from its description: xor-shift 16, multiply, xor-shift 13, multiply, xor-shift 16.
  Pinned by the published MurmurHash3_x86_32 vectors for the empty input.
* ``salt = fmix32(seed ^ fmix32(rank ^ fmix32(round)))``; ``h = fmix32(uint32(row*N + col) ^
  salt)`` with ``row`` local to the rank's slice (index taken modulo 2**32).
  Parity unpinned: no page fixes this composition.
* ``u = ((h >> 8) - 2**23) * 2**-23`` in float32 -- exact, and uniform on [-1, 1).
* bf16 = float32 rounded to nearest even (bit arithmetic); fp32 keeps ``u``; uint8 is
  ``h & 0xFF``.
"""
from __future__ import annotations

import numpy as np

_U32 = np.uint32


def fmix32(h) -> np.ndarray:
    """MurmurHash3 32-bit finaliser on a uint32 array (wrapping multiplies)."""
    h = np.array(h, dtype=np.uint32, copy=True, ndmin=1)
    with np.errstate(over="ignore"):
        h ^= h >> _U32(16)
        h *= _U32(0x85EBCA6B)
        h ^= h >> _U32(13)
        h *= _U32(0xC2B2AE35)
        h ^= h >> _U32(16)
    return h


def salt(seed: int, rank: int, rnd: int) -> int:
    """Per (seed, rank, round) salt: three nested finaliser applications."""
    a = fmix32(rnd & 0xFFFFFFFF)[0]
    b = fmix32((rank & 0xFFFFFFFF) ^ int(a))[0]
    return int(fmix32((seed & 0xFFFFFFFF) ^ int(b))[0])


def hash_at(seed: int, rank: int, rnd: int, rows, cols, N: int) -> np.ndarray:
    """uint32 hash for elements (rows[i], cols[i]) of a rank slice with N columns."""
    rows = np.asarray(rows, dtype=np.uint64)
    cols = np.asarray(cols, dtype=np.uint64)
    idx = (rows * np.uint64(N) + cols) & np.uint64(0xFFFFFFFF)
    return fmix32(idx.astype(np.uint32) ^ _U32(salt(seed, rank, rnd))).reshape(idx.shape)


def uniform_from_hash(h: np.ndarray) -> np.ndarray:
    """float32 value ((h >> 8) - 2**23) * 2**-23: exact, in [-1, 1)."""
    k = (np.asarray(h, dtype=np.uint32) >> _U32(8)).astype(np.int64) - (1 << 23)
    return (k.astype(np.float32) * np.float32(2.0 ** -23)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, nearest-even, by bit arithmetic (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return (r & np.uint64(0xFFFF)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << _U32(16)).view(np.float32)


def values_at(dtype: str, seed: int, rank: int, rnd: int, rows, cols, N: int) -> np.ndarray:
    """Element values in their storage type: uint16 bf16 bits, float32 or uint8."""
    h = hash_at(seed, rank, rnd, rows, cols, N)
    if dtype == "u8":
        return (h & _U32(0xFF)).astype(np.uint8)
    u = uniform_from_hash(h)
    if dtype == "f32":
        return u
    if dtype == "bf16":
        return f32_to_bf16_bits(u)
    raise ValueError(f"unknown dtype {dtype}")


def fill_slice(dtype: str, seed: int, rank: int, rnd: int, M: int, N: int) -> np.ndarray:
    """The [M, N] slice a producer writes in round ``rnd`` (storage type, row-major)."""
    rows = np.repeat(np.arange(M, dtype=np.uint64), N)
    cols = np.tile(np.arange(N, dtype=np.uint64), M)
    return values_at(dtype, seed, rank, rnd, rows, cols, N).reshape(M, N)


def fill_slice_bytes(dtype: str, seed: int, rank: int, rnd: int, M: int, N: int) -> np.ndarray:
    """Same as ``fill_slice`` viewed as raw little-endian bytes (uint8, length M*N*elem)."""
    return np.ascontiguousarray(fill_slice(dtype, seed, rank, rnd, M, N)).view(np.uint8).reshape(-1)
