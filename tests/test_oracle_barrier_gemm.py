"""Pins for the oracle's barrier (oracle/barrier.py) and GEMM reference (oracle/gemm.py)."""
import os

import numpy as np
import pytest

from oracle import barrier as B
from oracle import gemm as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    return [l for l in open(os.path.join(GOLDEN, name)) if l.strip() and not l.startswith("#")]


def test_handrolled_barrier_golden_columns():
    for line in _rows("barrier_columns.txt"):
        head, vals = line.split(":")
        P, r = (int(x) for x in head.split())
        want = np.array([int(x) for x in vals.split()])
        sig = np.zeros((P, P), dtype=np.int64)
        y = B.handrolled(sig, gen=1)
        assert np.array_equal(y[r], want)
        assert np.array_equal(B.expected_column(P, r), want)


def test_handrolled_barrier_reuse_with_generation_threshold():
    P = 5
    sig = np.zeros((P, P), dtype=np.int64)
    for gen in (1, 2, 3):
        y = B.handrolled(sig, gen=gen)
        for r in range(P):
            assert np.array_equal(y[r], B.expected_column(P, r, gen))


def test_reveal_golden():
    for line in _rows("reveal_p4.txt"):
        xs, ys = line.split(";")
        x = np.array([int(v) for v in xs.split()])[:, None]
        y = np.array([int(v) for v in ys.split()])[:, None]
        assert np.array_equal(B.reveal(x), y)
    x = np.arange(8 * 256).reshape(8, 256)
    y = B.reveal(x)
    assert all(np.array_equal(y[r], x[(r + 1) % 8]) for r in range(8))


def test_shared_cell_pitfall():
    P = 4
    # Set/Eq on one shared cell passes once a single peer has arrived ...
    assert B.shared_cell_set_eq([2], P)
    # ... AtomicAdd/Ge waits until every rank has arrived
    assert not B.shared_cell_add_ge([2], P)
    assert not B.shared_cell_add_ge([0, 1, 2], P)
    assert B.shared_cell_add_ge([0, 1, 2, 3], P)


def test_gemm_product_brute_force():
    rng = np.random.default_rng(0)
    A = rng.standard_normal((5, 7))
    Bt = rng.standard_normal((3, 7))
    C = G.product(A, Bt)
    for i in range(5):
        for j in range(3):
            acc = 0.0
            for k in range(7):
                acc += A[i, k] * Bt[j, k]
            assert abs(C[i, j] - acc) < 1e-12
    # identity and a rank-one product
    assert np.allclose(G.product(np.eye(4), np.eye(4)), np.eye(4))
    u, v = np.arange(1.0, 4.0), np.arange(2.0, 6.0)
    assert np.array_equal(G.product(u[:, None], v[:, None]), np.outer(u, v))


def test_rel_frobenius_closed_forms():
    C = np.arange(1.0, 13.0).reshape(3, 4)
    assert G.rel_frobenius(C, C) == 0.0
    assert G.rel_frobenius(np.zeros_like(C), C) == 1.0
    assert abs(G.rel_frobenius(1.01 * C, C) - 0.01) < 1e-12
    # one element off by d: d / ||C||_F
    D = C.copy()
    D[1, 2] += 0.5
    assert abs(G.rel_frobenius(D, C) - 0.5 / np.sqrt((C ** 2).sum())) < 1e-15


def test_bf16_bits_to_f64():
    assert G.bf16_bits_to_f64(np.array([0x3F80, 0xBF80, 0x4000, 0x0000], dtype=np.uint16)).tolist() \
        == [1.0, -1.0, 2.0, 0.0]
