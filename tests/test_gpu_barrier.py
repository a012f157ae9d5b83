"""GPU: the N-rank notify/wait barrier and the builtin reveal against the page's golden values
and the oracle."""
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import barrier as OB

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _windows(P):
    return ([torch.zeros(P, dtype=torch.int32, device="cuda") for _ in range(P)],
            [torch.full((P,), -7, dtype=torch.int32, device="cuda") for _ in range(P)],
            torch.full((P,), 99, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_handrolled_barrier_golden_and_reuse(P):
    sig, y, status = _windows(P)
    osig = np.zeros((P, P), dtype=np.int64)
    for gen in (1, 2, 3):
        D.dtt_barrier_handrolled(sig, y, gen, 1 << 24, status)
        torch.cuda.synchronize()
        oy = OB.handrolled(osig, gen)
        assert status.cpu().tolist() == [0] * P
        for r in range(P):
            assert y[r].cpu().tolist() == oy[r].tolist() == OB.expected_column(P, r, gen).tolist()
    golden = [l for l in open(os.path.join(GOLDEN, "barrier_columns.txt")) if l[0].isdigit()]
    sig, y, status = _windows(P)
    D.dtt_barrier_handrolled(sig, y, 1, 1 << 24, status)
    torch.cuda.synchronize()
    for line in golden:
        head, vals = line.split(":")
        gp, r = (int(x) for x in head.split())
        if gp == P:
            assert y[r].cpu().tolist() == [int(v) for v in vals.split()]


def test_handrolled_barrier_wait_gives_up():
    P = 4
    sig, y, status = _windows(P)
    D.dtt_barrier_handrolled(sig, y, 3, 2000, status)    # threshold nobody reaches
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [D.ETIMEDOUT] * P
    for r in range(P):
        assert y[r].cpu().tolist() == OB.expected_column(P, r, 1).tolist()


@pytest.mark.parametrize("P,size", [(8, 256), (2, 1), (5, 1000)])
def test_reveal(P, size):
    x_np = W.barrier_payload(P, size, seed=P * 1000 + size)
    x = [torch.from_numpy(x_np[r].copy()).cuda() for r in range(P)]
    data = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    y = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    status = torch.full((P,), 99, dtype=torch.int32, device="cuda")
    sig, ysig, _ = _windows(P)
    b = D.Barrier(P)
    try:
        for _ in range(3):                        # the internal counters' generations advance
            b.reveal(x, data, y, size, 1 << 24, status)
            torch.cuda.synchronize()
            assert status.cpu().tolist() == [0] * P
            want = OB.reveal(x_np)
            for r in range(P):
                np.testing.assert_array_equal(y[r].cpu().numpy(), want[r])
                np.testing.assert_array_equal(data[r].cpu().numpy(), x_np[r])
        assert all(int(s.abs().sum()) == 0 for s in sig)   # no tally in any user window
    finally:
        b.destroy()


def test_prepared_arguments_give_the_same_barriers():
    # arguments checked and marshalled once (HandrolledArgs / RevealArgs), reused call after
    # call: the same results as the list form, the page's columns and reveal
    P, size = 8, 64
    sig = [torch.zeros(P, dtype=torch.int32, device="cuda") for _ in range(P)]
    y = [torch.zeros(P, dtype=torch.int32, device="cuda") for _ in range(P)]
    status = torch.full((P,), 99, dtype=torch.int32, device="cuda")
    ha = D.HandrolledArgs(sig, y, status)
    osig = np.zeros((P, P), dtype=np.int64)          # the oracle's windows, across generations
    for gen in (1, 2, 3):
        D.dtt_barrier_handrolled(ha, gen=gen, max_polls=1 << 24)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0] * P
        want = OB.handrolled(osig, gen)
        for r in range(P):
            assert y[r].cpu().tolist() == want[r].tolist()
    x_np = W.barrier_payload(P, size, seed=3)
    x = [torch.from_numpy(x_np[r].copy()).cuda() for r in range(P)]
    data = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    yr = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    ra = D.RevealArgs(x, data, yr, size, status)
    b = D.Barrier(P)
    try:
        for _ in range(3):
            b.reveal(ra, max_polls=1 << 24)
            torch.cuda.synchronize()
            assert status.cpu().tolist() == [0] * P
            want = OB.reveal(x_np)
            for r in range(P):
                np.testing.assert_array_equal(yr[r].cpu().numpy(), want[r])
    finally:
        b.destroy()
