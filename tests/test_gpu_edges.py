"""GPU edges against the oracle: the largest plan (16 virtual ranks) on every transport, and a
chunk in more groups than the copier's signal keeps in registers."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import oracle_plan, oracle_round
from oracle import plan as OP

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner

TRANSPORTS = {"vector": dict(method=0, copier_threads=128),
              "bulk": dict(method=1, piece_bytes=8192, stages=2),
              "copy_engines": dict(method=2)}


def _rounds(w, opts, rounds, groups=None, **launch):
    st = runner.make(w, opts=opts, **launch)
    o = oracle_plan(w)
    if groups is not None:
        st.plan.define_groups(groups)
        o.define_groups(groups)
    try:
        for R in range(1, rounds + 1):
            rep = runner.run_round(st)
            assert rep.status == D.OK and rep.copier_timeouts == 0
            assert oracle_round(o, w) == (OP.OK, [], [])
            for q in range(w.P):
                np.testing.assert_array_equal(st.bufs[q].cpu().numpy(), o.bufs[q], err_msg=f"R{R} buffer {q}")
            np.testing.assert_array_equal(st.plan.read_gates()[:, :, :5], o.gates)
            if groups is not None:
                np.testing.assert_array_equal(st.plan.read_group_counters(), o.group_counters)
            st.plan.next_round()
            o.next_round()
    finally:
        st.plan.close()


@pytest.mark.parametrize("transport", sorted(TRANSPORTS))
def test_sixteen_ranks(transport):
    # DTT_MAX_RANKS virtual ranks, 2D tiles with ragged edges, every chunk to 15 peers
    w = W.Workload("p16", P=16, M=48, N=72, dtype=W.BF16, kind="tile_chunks", rounds=2, seed=161,
                   BM=16, BN=32, num_programs=3, tiles_per_chunk=3, group_m=2)
    _rounds(w, D.dtt_plan_opts_default(**TRANSPORTS[transport]), 2)


@pytest.mark.parametrize("transport", sorted(TRANSPORTS))
def test_chunk_in_many_groups(transport):
    # chunk 0 belongs to seven groups (more than the signal's register fast path holds); every
    # rank's counters equal the oracle's after each round
    w = W.small(W.C2, P=3, M=48, N=256, num_chunks=4)
    G = w.P * 4
    groups = [[0] + [g for g in range(1, G) if g % k == 0] for k in range(1, 8)] + [[c] for c in range(G)]
    _rounds(w, D.dtt_plan_opts_default(**TRANSPORTS[transport]), 3, groups=groups)
