"""GPU: the tcgen05 GEMM producer (C_r = A_r . B per virtual rank) feeding the triggered
all-gather.  The product is checked against the oracle's fp64 product of the same bf16
operands (relative Frobenius error <= 1e-2), every copy of C bit for bit against the rank's
own C, and the gates against the oracle's plan for the same tile_chunks schedule."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import oracle_plan
from oracle import gemm as OG
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner

TOL = 1e-2


def _slice(st, q, r):
    w = st.w
    S = w.slice_bytes
    return st.bufs[q][r * S:(r + 1) * S].view(torch.bfloat16).view(w.M, w.N)


def _oracle_gates_after(w, rounds):
    o = oracle_plan(w, copy_data=False)
    for rnd in range(rounds):
        o.start()
        for r in range(w.P):
            for c in o.chunks_of(r):
                for _ in range(o.chunks[c].writers):
                    o.mark_ready(r, c)
        o.copier_progress()
        assert o.wait()[0] == OP.OK
        if rnd < rounds - 1:
            o.next_round()
    return o


def _check(st, A, Bt, rows=None):
    w = st.w
    Bt64 = Bt.to(torch.float64).numpy()
    for r in range(w.P):
        mine = _slice(st, r, r)
        for q in range(w.P):                 # every copy equals the rank's own C, bit for bit
            assert torch.equal(_slice(st, q, r).view(torch.int16), mine.view(torch.int16)), (q, r)
        sel = slice(None) if rows is None else rows
        got = mine[sel].to(torch.float64).cpu().numpy()
        ref = OG.product(A[r][sel].to(torch.float64).numpy(), Bt64)
        err = OG.rel_frobenius(got, ref)
        assert err <= TOL, (r, err)
        assert err < 5e-3          # bf16 output rounding alone is about 2e-3


@pytest.mark.parametrize("P,M,N,K,NP", [
    # one-CTA form (M or N not a multiple of 256, or a single program)
    (2, 256, 384, 512, 5), (3, 128, 128, 64, 1), (2, 384, 256, 1024, 4),
    # CTA-pair form: one k-block, an odd program count, an idle pair, a single pair
    (1, 256, 256, 64, 2), (2, 768, 768, 192, 5), (3, 512, 256, 256, 8), (2, 256, 512, 512, 2)])
def test_gemm_producer_small(P, M, N, K, NP):
    w = W.Workload("g", P=P, M=M, N=N, dtype=W.BF16, kind="tile_chunks", rounds=2, seed=31 + M,
                   BM=128, BN=128, num_programs=NP, tiles_per_chunk=NP, K=K)
    A, Bt = W.gemm_inputs(P, M, N, K, w.seed)
    st = runner.make_gemm(w, A, Bt)
    try:
        for R in (1, 2):
            rep = runner.run_gemm_round(st)
            assert rep.status == D.OK and int(st.err.item()) == 0
            _check(st, A, Bt)
            o = _oracle_gates_after(st.w, R)
            np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
            st.plan.next_round()
    finally:
        st.plan.close()


def test_gemm_producer_full_size():
    w = W.C5
    A, Bt = W.gemm_inputs(w.P, w.M, w.N, w.K, w.seed)
    st = runner.make_gemm(w, A, Bt, opts=runner.bench_launch(w)["opts"])    # the benchmark's launch
    try:
        for R in range(1, 3):
            rep = runner.run_gemm_round(st)
            assert rep.status == D.OK and int(st.err.item()) == 0
            _check(st, A, Bt)            # all 2048 rows of every rank, every copy bit for bit
            st.plan.next_round()
    finally:
        st.plan.close()
