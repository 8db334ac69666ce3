"""Inputs of more than 2^31 elements (64-bit indexing everywhere): the
weighted sum on fp16 x[2^26 + 3, 40] (2.7e9 elements) and the scaled SiLU on
n = 2^31 + 2^20 + 5 fp16 elements (a ragged tail of 5).  Elementwise outputs
are compared on sampled rows / elements (boundaries, the tail, and seeded
random picks); grad_w and dw are compared complete — the oracle sums dw over
chunks of 2^28 elements (pairwise within a chunk, the chunk sums added in
fp64), whose error is far below the tolerance."""
import numpy as np
import pytest
import torch

import inputgen
import oracle
from inputgen import NORMAL, UNIFORM
from tolerance import GRAD_TOL, TOL, check_elementwise, check_reduction

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def test_ws_more_than_2_31_elements(wsf):
    N, D = (1 << 26) + 3, 40
    assert N * D > 2 ** 31
    x = inputgen.make((N, D), "f16", UNIFORM, -1.0, 1.0, 7, 0, pin=True)
    w = inputgen.make((D,), "f32", NORMAL, 0.0, 1.0, 7, 1)
    dy = inputgen.make((N,), "f16", NORMAL, 0.0, 1.0, 7, 2, pin=True)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    y = wsf.ws_fwd(xd, wd)
    dx, gw = wsf.ws_bwd(xd, wd, dyd)
    torch.cuda.synchronize()
    del xd
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, N // 2, N - 3, N - 2, N - 1], rng.choice(N, 4000)]))
    rt = torch.from_numpy(rows)
    xs, dys = x[rt].contiguous(), dy[rt].contiguous()
    ye, ya, yo = oracle.ws_fwd(xs, w)
    res = check_reduction(y[rt.to(DEV)].cpu(), ye, ya, D, TOL[torch.float16], ref_rounded=yo)
    assert res, ("y", res)
    r = oracle.ws_bwd(xs, w, dys)
    res = check_elementwise(dx[rt.to(DEV)].cpu(), r["dx"], np.outer(dys.double().numpy(), w.double().numpy()))
    assert res and res.clause2 == 0, ("dx", res)
    full = oracle.ws_bwd(x, w, dy, want_dx=False)
    res = check_reduction(gw.cpu(), full["grad_w"], full["grad_w_abs"], N, GRAD_TOL)
    assert res and res.clause2 == 0, ("grad_w", res)


def test_silu_more_than_2_31_elements(wsf):
    n = (1 << 31) + (1 << 20) + 5
    x = inputgen.make((n,), "f16", NORMAL, 0.0, 2.0, 8, 0, pin=True)
    dy = inputgen.make((n,), "f16", NORMAL, 0.0, 1.0, 8, 2, pin=True)
    w = torch.tensor([0.75], dtype=torch.float32)
    xd, dyd, wd = x.to(DEV), dy.to(DEV), w.to(DEV)
    y = wsf.silu_fwd(xd, wd)
    dx, dw = wsf.silu_bwd(dyd, xd, wd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    idx = np.unique(np.concatenate([np.arange(8), np.arange(n - 64, n), [2 ** 31 - 1, 2 ** 31, 2 ** 31 + 1],
                                    rng.choice(n, 200000)]))
    it = torch.from_numpy(idx)
    xs, gs = x[it].contiguous(), dy[it].contiguous()
    ye, yo = oracle.silu_fwd(xs, 0.75)
    res = check_elementwise(y[it.to(DEV)].cpu(), yo, ye)
    assert res, ("y", res)
    ro = oracle.silu_bwd(gs, xs, 0.75, want_dw=False)
    res = check_elementwise(dx[it.to(DEV)].cpu(), ro["dx"], ro["dx_exact"], scale=ro["dx_scale"])
    assert res, ("dx", res)
    del xd, dyd, y, dx
    total, total_abs = 0.0, 0.0
    step = 1 << 28
    for a in range(0, n, step):
        rc = oracle.silu_bwd(dy[a:a + step], x[a:a + step], 0.75, want_dx=False)
        total += rc["dw"]
        total_abs += rc["dw_abs"]
    res = check_reduction(dw.cpu(), np.array([total]), np.array([total_abs]), n, GRAD_TOL)
    assert res, ("dw", res)
