"""Failure detection of the cluster exchange, without a GPU fault: the bounded
wait that the cluster paths use gives up when the partial sums it waits for
never arrive (an mbarrier turn that no CTA pushes to), counts one timeout for
each waiting warp in a device counter the host reads, and leaves the context
usable — a cluster-path softmax launched afterwards still matches the oracle."""
import time

import pytest
import torch

import oracle
from tolerance import check_elementwise

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def test_exchange_wait_runs_out_and_context_stays_usable(wsf):
    before = wsf.cluster_wait_timeouts()
    count = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    wsf.selftest_exchange_timeout(count, limit_ms=20)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    warps = wsf.selftest_waiting_warps()
    assert int(count.item()) == warps
    assert 0.02 <= dt < 5.0, dt
    # a second run adds as many again
    wsf.selftest_exchange_timeout(count, limit_ms=5)
    torch.cuda.synchronize()
    assert int(count.item()) == 2 * warps
    # the library's own counter is untouched, and the device still computes
    assert wsf.cluster_wait_timeouts() == before
    import inputgen
    from inputgen import NORMAL
    x = inputgen.make((8, 50000), "bf16", NORMAL, 0.0, 2.0, 0, 0)
    y = wsf.softmax_fwd(x.to(DEV))
    torch.cuda.synchronize()
    ye, yo = oracle.softmax_fwd(x)
    res = check_elementwise(y.cpu(), yo, ye)
    assert res, res
    assert wsf.cluster_wait_timeouts() == before
