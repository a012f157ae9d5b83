"""GPU: the reveal barrier's entry point that allocates nothing, checked against the
allocating entry point.  Some callers cannot allocate device memory when they call the
library (their memory belongs to another allocator, or they cannot afford the device-wide
synchronisation that cudaFree brings); dtt_barrier_reveal_noalloc keeps its counters in a fixed
device array instead.  Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from conftest import ensure_built
    ensure_built()
    import device_triggered_transfers_gb300 as D


def _slices(P, size, fill=0):
    return [torch.full((size,), fill, dtype=torch.int32, device="cuda") for _ in range(P)]


def test_noalloc_reveal_matches_allocating_reveal_on_two_calls():
    P, size = 8, 256
    b = D.Barrier(P)
    data_a, y_a, data_b, y_b = (_slices(P, size, -1) for _ in range(4))
    st_a = torch.full((P,), 99, dtype=torch.int32, device="cuda")
    st_b = torch.full((P,), 99, dtype=torch.int32, device="cuda")
    try:
        for call in range(2):                      # the array keeps the last call's counts
            x_np = W.barrier_payload(P, size, seed=1000 + call)
            x = [torch.from_numpy(x_np[r].copy()).cuda() for r in range(P)]
            torch.cuda.synchronize()
            D.dtt_barrier_reveal_noalloc(x, data_b, y_b, size, 1 << 24, st_b)
            b.reveal(x, data_a, y_a, size, 1 << 24, st_a)
            torch.cuda.synchronize()
            assert st_b.cpu().tolist() == [0] * P
            assert st_a.cpu().tolist() == [0] * P
            for r in range(P):
                assert torch.equal(y_b[r], y_a[r]), (call, r)
                assert torch.equal(data_b[r], data_a[r]), (call, r)
                np.testing.assert_array_equal(y_b[r].cpu().numpy(), x_np[(r + 1) % P])
    finally:
        b.destroy()


def test_noalloc_reveal_rejects_more_ranks_than_its_array_holds():
    P = 17
    s = _slices(P, 4)
    with pytest.raises(D.DttError) as e:
        D.dtt_barrier_reveal_noalloc(s, s, s, 4, 100, torch.zeros(P, dtype=torch.int32, device="cuda"))
    assert e.value.code == D.EINVAL
