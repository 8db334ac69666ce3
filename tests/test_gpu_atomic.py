"""The atomic comparison variants: same results as the two-pass kernels up
to fp32 rounding (checked against the oracle), identical dx, and a count of
how many distinct bit patterns the parameter gradient takes over repeated
runs (the two-pass form must always give exactly one)."""
import numpy as np
import pytest
import torch

import oracle
from inputgen import NORMAL
from tolerance import GRAD_TOL, check_reduction

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def _patterns(ts):
    return len({bytes(t.view(torch.int32).cpu().numpy()) for t in ts})


@pytest.mark.parametrize("N,D,dt", [(200_003, 64, "f16"), (20_000, 1024, "bf16"), (64, 8200, "f32")])
def test_ws_bwd_atomic(wsf, N, D, dt):
    import inputgen
    x = inputgen.make((N, D), dt, NORMAL, 0, 1, 0, 0)
    w = inputgen.make((D,), "f32", NORMAL, 0, D ** -0.5, 0, 1)
    dy = inputgen.make((N,), dt, NORMAL, 0, 1, 0, 2)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    dx_ref, gw_ref = wsf.ws_bwd(xd, wd, dyd)
    runs = [wsf.ws_bwd_atomic(xd, wd, dyd) for _ in range(8)]
    two = [wsf.ws_bwd(xd, wd, dyd)[1] for _ in range(4)]
    torch.cuda.synchronize()
    r = oracle.ws_bwd(x, w, dy, want_dx=False)
    for dx, gw in runs:
        assert torch.equal(dx, dx_ref)
        assert check_reduction(gw.cpu(), r["grad_w"], r["grad_w_abs"], N, GRAD_TOL)
    assert _patterns(two) == 1
    print(f"ws {N}x{D} {dt}: atomic grad_w took {_patterns([g for _, g in runs])} bit patterns in 8 runs")
    acc = gw_ref.clone()
    wsf.ws_bwd_atomic(xd, wd, dyd, grad_w=acc, accumulate=True)
    assert check_reduction((acc - gw_ref).cpu(), r["grad_w"], r["grad_w_abs"], N, 1e-4)


def test_silu_bwd_atomic(wsf):
    import inputgen
    n = 8192 * 512 + 5
    x = inputgen.make((n,), "f16", NORMAL, 0, 2, 0, 0)
    dy = inputgen.make((n,), "f16", NORMAL, 0, 1, 0, 2)
    w = torch.tensor([0.75], device=DEV)
    xd, gd = x.to(DEV), dy.to(DEV)
    dx_ref, _ = wsf.silu_bwd(gd, xd, w)
    runs = [wsf.silu_bwd_atomic(gd, xd, w) for _ in range(8)]
    torch.cuda.synchronize()
    r = oracle.silu_bwd(dy, x, 0.75, want_dx=False)
    for dx, dw in runs:
        assert torch.equal(dx, dx_ref)
        assert check_reduction(np.array([float(dw)]), np.array([r["dw"]]), np.array([r["dw_abs"]]),
                               n, GRAD_TOL)
    print(f"silu n={n}: atomic dw took {_patterns([d for _, d in runs])} bit patterns in 8 runs")
    # misaligned pointers take the scalar kernel, also atomic
    xb = torch.zeros(n + 1, dtype=torch.float16, device=DEV)
    xb[1:].copy_(xd)
    _, dwm = wsf.silu_bwd_atomic(gd, xb[1:], w)
    torch.cuda.synchronize()
    assert check_reduction(np.array([float(dwm)]), np.array([r["dw"]]), np.array([r["dw_abs"]]),
                           n, GRAD_TOL)


def test_ws_bwd_atomic_rejects_unaligned(wsf):
    x = torch.zeros((10, 60), dtype=torch.float16, device=DEV)
    with pytest.raises(wsf.WsfError) as e:
        wsf.ws_bwd_atomic(x, torch.zeros(60, device=DEV), torch.zeros(10, dtype=torch.float16,
                                                                      device=DEV))
    assert e.value.status == wsf.ERR_MISALIGNED
