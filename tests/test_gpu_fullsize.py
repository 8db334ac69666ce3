"""Full-size workloads (the benchmark's sizes and launch configuration)
against the oracle: y and dx on sampled rows (first, last, middle and 4,090
seeded random rows), grad_w / dw complete, and grad_w bit-identical across
two runs.  The scaled-SiLU workload is compared element by element."""
import numpy as np
import pytest
import torch

import inputgen
import oracle
from inputgen.workloads import WORKLOADS
from tolerance import GRAD_TOL, TOL, check_elementwise, check_reduction

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def host_inputs(wl):
    x = inputgen.make((wl.N, wl.D), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0, pin=True)
    w = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1)
    dy = inputgen.make((wl.N,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2, pin=True)
    return x, w, dy


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_ws_full_size(wsf, name):
    wl = WORKLOADS[name]
    x, w, dy = host_inputs(wl)
    xd, wd, dyd = x.to(DEV, non_blocking=True), w.to(DEV), dy.to(DEV, non_blocking=True)
    y = wsf.ws_fwd(xd, wd)
    dx, gw = wsf.ws_bwd(xd, wd, dyd)
    _, gw2 = wsf.ws_bwd(xd, wd, dyd, dx=torch.empty_like(dx))
    torch.cuda.synchronize()
    assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32)), "grad_w not bit-reproducible"
    rng = np.random.default_rng(0)
    N = wl.N
    rows = np.unique(np.concatenate([[0, 1, 2, N // 2, N - 2, N - 1], rng.choice(N, 4090)]))
    rt = torch.from_numpy(rows)
    xs, dys = x[rt].contiguous(), dy[rt].contiguous()
    ye, ya, yo = oracle.ws_fwd(xs, w)
    res = check_reduction(y[rt.to(DEV)].cpu(), ye, ya, wl.D, TOL[x.dtype], ref_rounded=yo)
    assert res, ("y", res)
    r = oracle.ws_bwd(xs, w, dys)
    exact_dx = np.outer(dys.double().numpy(), w.double().numpy())
    res = check_elementwise(dx[rt.to(DEV)].cpu(), r["dx"], exact_dx)
    assert res and res.clause2 == 0, ("dx", res)
    full = oracle.ws_bwd(x, w, dy, want_dx=False)
    res = check_reduction(gw.cpu(), full["grad_w"], full["grad_w_abs"], N, GRAD_TOL)
    # compensated sums: every column within 1e-5 of the exact value, none
    # passing only by the cancellation clause
    assert res and res.clause2 == 0, ("grad_w", res)


def test_silu_full_size(wsf):
    wl = WORKLOADS["c2"]
    n = wl.n
    x = inputgen.make((n,), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0, pin=True)
    dy = inputgen.make((n,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2, pin=True)
    w = torch.tensor([wl.w_scalar])
    xd, gd, wd = x.to(DEV), dy.to(DEV), w.to(DEV)
    y = wsf.silu_fwd(xd, wd)
    dx, dw = wsf.silu_bwd(gd, xd, wd)
    _, dw2 = wsf.silu_bwd(gd, xd, wd, dx=torch.empty_like(dx))
    torch.cuda.synchronize()
    assert torch.equal(dw.view(torch.int32), dw2.view(torch.int32)), "dw not bit-reproducible"
    ye, yo = oracle.silu_fwd(x, wl.w_scalar)
    res = check_elementwise(y.cpu(), yo, ye)
    assert res and res.clause2 == 0, ("y", res)
    r = oracle.silu_bwd(dy, x, wl.w_scalar)
    res = check_elementwise(dx.cpu(), r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert res and res.clause2 == 0, ("dx", res)
    res = check_reduction(np.array([float(dw)]), np.array([r["dw"]]), np.array([r["dw_abs"]]), n,
                          GRAD_TOL)
    assert res and res.clause2 == 0, ("dw", res, float(dw), r["dw"])
