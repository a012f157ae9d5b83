"""Pins for the oracle's producer values (oracle/hashfill.py), independent of the oracle."""
import os

import numpy as np
import pytest
import torch

from oracle import hashfill as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_fmix32_published_murmur3_vectors():
    # MurmurHash3_x86_32 of the empty input reduces to fmix32(seed); its published test vectors
    # are 0 for seed 0, 0x514E28B7 for seed 1 and 0x81F16F39 for seed 0xFFFFFFFF.
    assert int(H.fmix32(0)[0]) == 0
    assert int(H.fmix32(1)[0]) == 0x514E28B7
    assert int(H.fmix32(0xFFFFFFFF)[0]) == 0x81F16F39


def test_fmix32_vectorised_matches_scalar_calls():
    x = np.arange(1000, dtype=np.uint32) * np.uint32(2654435761)
    v = H.fmix32(x)
    for i in (0, 1, 17, 999):
        assert v[i] == H.fmix32(int(x[i]))[0]


def test_uniform_is_exact_and_in_range():
    h = np.array([0, 0xFF, 0x100, 0x80000000, 0xFFFFFFFF, 0x7FFFFF00], dtype=np.uint32)
    u = H.uniform_from_hash(h)
    # closed form: ((h >> 8) - 2**23) / 2**23
    want = [((int(x) >> 8) - (1 << 23)) / float(1 << 23) for x in h]
    assert u.dtype == np.float32
    assert list(u.astype(np.float64)) == want
    assert u.min() == -1.0 and u.max() == 1.0 - 2.0 ** -23
    r = H.uniform_from_hash(np.random.default_rng(0).integers(0, 1 << 32, 100000, dtype=np.uint64)
                            .astype(np.uint32))
    assert np.all(r >= -1.0) and np.all(r < 1.0)
    assert np.all((r.astype(np.float64) * 2 ** 23) == np.round(r.astype(np.float64) * 2 ** 23))
    assert abs(float(r.mean())) < 0.01


def test_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = rng.uniform(-1, 1, 200000).astype(np.float32)
    # exact ties, and values one ulp either side of a tie
    base = (rng.integers(0, 1 << 15, 2000).astype(np.uint32) << np.uint32(16))
    ties = np.concatenate([base | np.uint32(0x8000), base | np.uint32(0x7FFF),
                           base | np.uint32(0x8001), base | np.uint32(0x18000)])
    x = np.concatenate([x, ties.view(np.float32), np.float32([0.0, -0.0, 1.0, -1.0])])
    x = x[np.isfinite(x)]
    ours = H.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_values_depend_on_round_rank_and_position():
    a = H.fill_slice("bf16", 7, 0, 1, 16, 32)
    assert not np.array_equal(a, H.fill_slice("bf16", 7, 0, 2, 16, 32))
    assert not np.array_equal(a, H.fill_slice("bf16", 7, 1, 1, 16, 32))
    assert not np.array_equal(a, H.fill_slice("bf16", 8, 0, 1, 16, 32))
    # bf16 has few values near +-1, so distinctness is checked on the fp32 form
    assert len(np.unique(H.fill_slice("f32", 7, 0, 1, 16, 32))) > 500


def test_dtypes_share_one_hash():
    h = H.hash_at(3, 2, 5, np.arange(64), np.arange(64), 1000)
    assert np.array_equal(H.values_at("u8", 3, 2, 5, np.arange(64), np.arange(64), 1000),
                          (h & 0xFF).astype(np.uint8))
    f = H.values_at("f32", 3, 2, 5, np.arange(64), np.arange(64), 1000)
    b = H.values_at("bf16", 3, 2, 5, np.arange(64), np.arange(64), 1000)
    assert np.array_equal(b, H.f32_to_bf16_bits(f))


def test_spot_table():
    """Regression pin: values written once by tests/golden/make_hash_spot.py (oracle only)."""
    path = os.path.join(GOLDEN, "hash_spot.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 20
    for dtype, seed, rank, rnd, row, col, N, val in rows:
        got = H.values_at(dtype, int(seed), int(rank), int(rnd), [int(row)], [int(col)], int(N))
        raw = got.view(np.uint8 if dtype == "u8" else (np.uint32 if dtype == "f32" else np.uint16))
        assert int(raw[0]) == int(val, 16), (dtype, seed, rank, rnd, row, col)


# ---- the plain-C restatement (oracle/cfill.py, oracle/fill.c): the same pins, then element-by-
# element agreement with the numpy restatement -----------------------------------------------
from oracle import cfill  # noqa: E402


def test_c_fmix32_published_murmur3_vectors():
    assert cfill.fmix32(0) == 0
    assert cfill.fmix32(1) == 0x514E28B7
    assert cfill.fmix32(0xFFFFFFFF) == 0x81F16F39


def test_c_uniform_is_exact_closed_form():
    for h in (0, 0xFF, 0x100, 0x80000000, 0xFFFFFFFF, 0x7FFFFF00, 0x12345678):
        u = np.uint32(cfill.uniform_bits(h)).view(np.float32)
        assert float(u) == ((h >> 8) - (1 << 23)) / float(1 << 23)


def test_c_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(2)
    x = rng.uniform(-1, 1, 20000).astype(np.float32)
    base = (rng.integers(0, 1 << 15, 500).astype(np.uint32) << np.uint32(16))
    ties = np.concatenate([base | np.uint32(0x8000), base | np.uint32(0x7FFF),
                           base | np.uint32(0x8001), base | np.uint32(0x18000)])
    x = np.concatenate([x, ties.view(np.float32), np.float32([0.0, -0.0, 1.0, -1.0])])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([cfill.bf16_bits(int(b)) for b in x.view(np.uint32)], dtype=np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "u8"])
def test_c_fill_equals_numpy_fill(dtype):
    # ragged shapes, several seeds / ranks / rounds, and an index past 2^32 (the mod 2^32 rule)
    for (seed, rank, rnd, M, N) in [(1, 0, 1, 7, 33), (20261202, 3, 9, 16, 1024),
                                    (0xFFFFFFFF, 15, 0xFFFFFFFF, 3, 5)]:
        a = cfill.fill_slice_bytes(dtype, seed, rank, rnd, M, N, threads=3)
        b = H.fill_slice_bytes(dtype, seed, rank, rnd, M, N)
        assert np.array_equal(a, b), (dtype, seed, rank, rnd)
    rows = np.array([(1 << 32) // 4096 + 5, 123456], dtype=np.uint64)
    N = 4096
    out = np.empty(N * {"bf16": 2, "f32": 4, "u8": 1}[dtype], dtype=np.uint8)
    for r in rows:
        cfill.fill_rows_into(out, dtype, 5, 2, 7, N, int(r), int(r) + 1)
        want = H.values_at(dtype, 5, 2, 7, np.full(N, r), np.arange(N), N)
        assert np.array_equal(out, np.ascontiguousarray(want).view(np.uint8))


def test_c_salt_matches_numpy_salt():
    for args in [(0, 0, 0), (20261202, 7, 10), (0xFFFFFFFF, 15, 0xFFFFFFFF)]:
        assert cfill.salt(*args) == H.salt(*args)


def test_expected_buffer_is_every_rank_slice_in_place():
    import workloads as W
    w = W.small(W.C2, M=8, N=64, num_chunks=2)
    buf = cfill.expected_buffer(w, 3)
    S = w.slice_bytes
    for r in range(w.P):
        assert np.array_equal(buf[r * S:(r + 1) * S], H.fill_slice_bytes(w.dtype, w.seed, r, 3, w.M, w.N))
    b = W.Workload("b", P=3, M=4, N=100, dtype=W.U8, kind="whole", rounds=1, seed=4, broadcast=True)
    assert np.array_equal(cfill.expected_buffer(b, 1), H.fill_slice_bytes("u8", 4, 0, 1, 4, 100))
