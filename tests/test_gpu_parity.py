"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Sizes span several tiles with ragged tails; the sweep covers every kernel
family (register, wide, tile and scalar paths), row strides, misaligned
pointers, block_n tilings, accumulation, empty inputs, integer inputs that
must match bit for bit, run-to-run bit reproducibility, guard bands around
every output, and the worked 100 x 64 / 32-row-tile shape.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from inputgen import NORMAL, UNIFORM
from tolerance import GRAD_TOL, TOL, check_elementwise, check_reduction

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTS = ["f32", "f16", "bf16"]
DEV = "cuda:0"
CANARY = 77  # byte pattern written around outputs


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    assert torch.cuda.is_available()
    return m


def guarded(shape, dtype, pad=256):
    """A device tensor view inside a larger byte buffer whose margins hold a
    canary pattern; returns (view, check) where check() asserts the margins
    are intact."""
    n = int(np.prod(shape)) if len(shape) else 1
    es = torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((n * es + 2 * pad,), CANARY, dtype=torch.uint8, device=DEV)
    view = buf[pad:pad + n * es].view(dtype).view(shape)

    def check():
        torch.cuda.synchronize()
        assert bool((buf[:pad] == CANARY).all()) and bool((buf[pad + n * es:] == CANARY).all()), \
            "write outside the output"
    return view, check


def make_ws(N, D, dt, seed_shift=0, xdist=(NORMAL, 0.0, 1.0)):
    import inputgen
    x = inputgen.make((N, D), dt, xdist[0], xdist[1], xdist[2], 0, 0 + seed_shift)
    w = inputgen.make((D,), "f32", NORMAL, 0.0, 1.0 / math.sqrt(max(D, 1)), 0, 1 + seed_shift)
    dy = inputgen.make((N,), dt, NORMAL, 0.0, 1.0, 0, 2 + seed_shift)
    return x, w, dy


def run_ws(wsf, x, w, dy, ld_pad=0, misalign=0, block_n=0, dy_misalign=None):
    """Place inputs on the device (optionally with a row stride of D + ld_pad
    and pointers shifted by `misalign` elements; dy alone by `dy_misalign`),
    run forward and backward with guarded outputs; returns host results."""
    N, D = x.shape
    dt = x.dtype
    ld = D + ld_pad
    dmis = misalign if dy_misalign is None else dy_misalign
    xb = torch.zeros(N * ld + misalign + 8, dtype=dt, device=DEV)
    xd = xb[misalign:misalign + N * ld].view(N, ld)[:, :D]
    xd.copy_(x.to(DEV))
    dyb = torch.zeros(N + dmis + 8, dtype=dt, device=DEV)
    dyd = dyb[dmis:dmis + N]
    dyd.copy_(dy.to(DEV))
    wd = w.to(DEV)
    y, ychk = guarded((N,), dt)
    wsf.ws_fwd(xd, wd, y=y)
    dxb, dxchk = guarded((N * ld + misalign,), dt)
    dx = dxb[misalign:].view(N, ld)[:, :D] if N * D > 0 else dxb[:0].view(N, D)
    gw, gwchk = guarded((D,), torch.float32)
    wsf.ws_bwd(xd, wd, dyd, dx=dx, grad_w=gw, block_n=block_n)
    ychk()
    dxchk()
    gwchk()
    return y.cpu(), dx.cpu(), gw.cpu()


def assert_ws_parity(x, w, dy, y, dx, gw):
    N, D = x.shape
    ye, ya, yo = oracle.ws_fwd(x, w)
    r = oracle.ws_bwd(x, w, dy)
    tol = TOL[x.dtype]
    res = check_reduction(y, ye, ya, D, tol, ref_rounded=yo)
    assert res, ("y", res)
    exact_dx = np.outer(dy.double().numpy(), w.double().numpy())
    res = check_elementwise(dx, r["dx"], exact_dx)
    assert res and res.clause2 == 0, ("dx", res)
    if x.dtype == torch.float32:
        assert torch.equal(dx, r["dx"])  # one fp32 rounding of an exact product on both sides
    # compensated sums: every column within 1e-5 of the exact value
    res = check_reduction(gw, r["grad_w"], r["grad_w_abs"], N, GRAD_TOL)
    assert res and res.clause2 == 0, ("grad_w", res)


WS_SHAPES = [(1, 1), (1, 64), (7, 5), (31, 63), (32, 64), (33, 65), (100, 64), (129, 8),
             (7, 1024), (33, 1000), (64, 1032), (5, 2048), (3, 2056), (9, 4097), (17, 8200),
             (2, 70000), (700, 16)]


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", WS_SHAPES)
def test_ws_parity_shapes(wsf, dt, N, D):
    x, w, dy = make_ws(N, D, dt)
    y, dx, gw = run_ws(wsf, x, w, dy)
    assert_ws_parity(x, w, dy, y, dx, gw)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D,ld_pad,misalign", [(37, 64, 8, 0), (37, 64, 3, 0), (37, 64, 0, 1),
                                                 (11, 1024, 8, 0), (11, 1000, 1, 1),
                                                 (5, 2056, 16, 0), (5, 2056, 0, 3)])
def test_ws_parity_strides_alignment(wsf, dt, N, D, ld_pad, misalign):
    x, w, dy = make_ws(N, D, dt)
    y, dx, gw = run_ws(wsf, x, w, dy, ld_pad=ld_pad, misalign=misalign)
    assert_ws_parity(x, w, dy, y, dx, gw)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(37, 64), (1000, 8), (77, 1024), (9, 2056), (5, 8200)])
def test_ws_parity_register_tile_path(wsf, dt, N, D):
    """x and dx 16-byte aligned but dy not: the backward uses the register-load
    tile kernel instead of the cp.async-staged one."""
    x, w, dy = make_ws(N, D, dt)
    y, dx, gw = run_ws(wsf, x, w, dy, dy_misalign=1)
    assert_ws_parity(x, w, dy, y, dx, gw)


@pytest.mark.parametrize("block_n", [1, 7, 32, 1000])
@pytest.mark.parametrize("dt", DTS)
def test_ws_block_n(wsf, dt, block_n):
    x, w, dy = make_ws(100, 64, dt)
    y, dx, gw = run_ws(wsf, x, w, dy, block_n=block_n)
    assert_ws_parity(x, w, dy, y, dx, gw)


def test_worked_shape_partial_buffer(wsf):
    """100 rows, D = 64, 32-row tiles: the workspace holds exactly the four
    partial rows (the last over rows 96..99), each as a compensated pair (a
    [4, 64] plane of high parts, then one of low parts), and grad_w is their
    sum."""
    x, w, dy = make_ws(100, 64, "f32")
    need = wsf.ws_bwd_workspace_bytes(100, 64, torch.float32, 32)
    assert need == 2 * 4 * 64 * 4
    ws = torch.full((need + 512,), CANARY, dtype=torch.uint8, device=DEV)
    _, gw = wsf.ws_bwd(x.to(DEV), w.to(DEV), dy.to(DEV), workspace=ws[:need], block_n=32)
    torch.cuda.synchronize()
    assert bool((ws[need:] == CANARY).all())
    planes = ws[:need].view(torch.float32).view(2, 4, 64).cpu().double()
    part = (planes[0] + planes[1]).numpy()
    r = oracle.ws_bwd(x, w, dy, block_n=32)
    for p in range(4):
        a, b = 32 * p, min(100, 32 * p + 32)
        ab = oracle.ws_bwd(x[a:b].contiguous(), w, dy[a:b].contiguous())["grad_w_abs"]
        res = check_reduction(part[p], r["partial"][p], ab, b - a, GRAD_TOL)
        assert res and res.clause2 == 0, (p, res)
    # stage 2: the four pairs summed in ascending order, rounded once
    res = check_reduction(gw.cpu(), r["grad_w"], r["grad_w_abs"], 100, GRAD_TOL)
    assert res and res.clause2 == 0, res


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(1, 1), (1, 64), (7, 5), (7, 64), (100, 64), (33, 1000),
                                 (3000, 8), (65, 2056), (9, 8200)])
def test_ws_integer_exact(wsf, dt, N, D):
    """x, w, dy in {-1, 0, 1}: all sums are small integers, exact in any
    order, so y, dx and grad_w must equal integer arithmetic bit for bit
    (batch 1 and batch 7 included: a missing batch reduction shows at 7)."""
    rng = np.random.default_rng(N * 7919 + D)
    xi, wi, gi = rng.integers(-1, 2, (N, D)), rng.integers(-1, 2, D), rng.integers(-1, 2, N)
    x = torch.from_numpy(xi.astype(np.float32)).to(TDT[dt])
    w = torch.from_numpy(wi.astype(np.float32))
    dy = torch.from_numpy(gi.astype(np.float32)).to(TDT[dt])
    for block_n in [0, 32]:
        y, dx, gw = run_ws(wsf, x, w, dy, block_n=block_n)
        # the fp32 sum is an exact integer; the store rounds it once to the type
        yref = torch.from_numpy((xi @ wi).astype(np.float32)).to(TDT[dt]).float().numpy()
        assert np.array_equal(y.float().numpy(), yref)
        assert np.array_equal(dx.float().numpy(), np.outer(gi, wi).astype(np.float32))
        assert np.array_equal(gw.numpy(), (xi.T @ gi).astype(np.float32))


@pytest.mark.parametrize("dt", DTS)
def test_ws_bit_reproducible(wsf, dt):
    x, w, dy = make_ws(5000, 1024 if dt != "f32" else 512, dt)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    outs = [wsf.ws_bwd(xd, wd, dyd) for _ in range(3)]
    ys = [wsf.ws_fwd(xd, wd) for _ in range(3)]
    torch.cuda.synchronize()
    for (dx, gw) in outs[1:]:
        assert torch.equal(dx, outs[0][0])
        assert torch.equal(gw.view(torch.int32), outs[0][1].view(torch.int32))
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


@pytest.mark.parametrize("dt", DTS)
def test_ws_accumulate(wsf, dt):
    """accumulate = 1 adds the batch gradient to grad_w with one fp32 add
    (gradients accumulate with += across micro-batches)."""
    x, w, dy = make_ws(300, 200, dt)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    g0 = torch.randn(200, generator=torch.Generator().manual_seed(3)).float()
    _, fresh = wsf.ws_bwd(xd, wd, dyd)
    acc = g0.to(DEV).clone()
    wsf.ws_bwd(xd, wd, dyd, grad_w=acc, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(acc.cpu(), g0 + fresh.cpu())


def test_ws_empty(wsf):
    w = torch.randn(16, device=DEV)
    x = torch.empty((0, 16), device=DEV)
    dy = torch.empty((0,), device=DEV)
    gw = torch.full((16,), 5.0, device=DEV)
    wsf.ws_bwd(x, w, dy, grad_w=gw)
    assert bool((gw == 0).all())
    gw.fill_(5.0)
    wsf.ws_bwd(x, w, dy, grad_w=gw, accumulate=True)
    assert bool((gw == 5.0).all())
    # D == 0: every row's empty sum is 0
    x0 = torch.empty((9, 0), device=DEV)
    y = torch.full((9,), 3.0, device=DEV)
    wsf.ws_fwd(x0, torch.empty(0, device=DEV), y=y)
    assert bool((y == 0).all())
    wsf.ws_fwd(torch.empty((0, 16), device=DEV), w, y=torch.empty(0, device=DEV))


def test_ws_rejects_on_device(wsf):
    x, w, dy = make_ws(100, 64, "f32")
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(wsf.WsfError) as e:
        wsf.ws_bwd(xd, wd, dyd, workspace=small)
    assert e.value.status == wsf.ERR_WORKSPACE
    with pytest.raises(wsf.WsfError) as e:
        wsf.ws_bwd(xd, wd, dyd, dx=xd)
    assert e.value.status == wsf.ERR_OVERLAP


def test_temporary_workspace_on_a_side_stream(wsf):
    """A workspace the binding allocates for a call on another stream must
    stay the call's until that stream has used it: a tensor allocated and
    filled on the default stream meanwhile must not share its memory."""
    x, w, dy = make_ws(20000, 1024, "bf16")
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    _, gw_ref = wsf.ws_bwd(xd, wd, dyd)
    need = wsf.ws_bwd_workspace_bytes(20000, 1024, torch.bfloat16)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)  # holds the side stream back for some milliseconds
    dx, gw = wsf.ws_bwd(xd, wd, dyd, stream=side)
    junk = torch.full((need // 4,), 1e30, dtype=torch.float32, device=DEV)
    side.synchronize()
    torch.cuda.synchronize()
    assert bool((junk == 1e30).all()), "the temporary workspace was handed out while in use"
    assert torch.equal(gw.view(torch.int32), gw_ref.view(torch.int32))


# ---------------------------------------------------------------------------- SiLU
def make_silu(n, dt, w=0.75):
    import inputgen
    x = inputgen.make((n,), dt, NORMAL, 0.0, 2.0, 0, 0)
    dy = inputgen.make((n,), dt, NORMAL, 0.0, 1.0, 0, 2)
    return x, dy, torch.tensor([w], dtype=torch.float32)


def run_silu(wsf, x, dy, w, misalign=0):
    n = x.numel()
    dt = x.dtype
    xb = torch.zeros(n + misalign + 8, dtype=dt, device=DEV)
    xd = xb[misalign:misalign + n]
    xd.copy_(x.to(DEV))
    gb = torch.zeros(n + misalign + 8, dtype=dt, device=DEV)
    gd = gb[misalign:misalign + n]
    gd.copy_(dy.to(DEV))
    wd = w.to(DEV)
    yb, ychk = guarded((n + misalign,), dt)
    y = yb[misalign:]
    wsf.silu_fwd(xd, wd, y=y)
    dxb, dxchk = guarded((n + misalign,), dt)
    dx = dxb[misalign:]
    dw, dwchk = guarded((1,), torch.float32)
    wsf.silu_bwd(gd, xd, wd, dx=dx, dw=dw)
    ychk()
    dxchk()
    dwchk()
    return y.cpu(), dx.cpu(), float(dw.cpu())


def assert_silu_parity(x, dy, w, y, dx, dw):
    ye, yo = oracle.silu_fwd(x, float(w))
    r = oracle.silu_bwd(dy, x, float(w))
    res = check_elementwise(y, yo, ye)
    assert res and res.clause2 == 0, ("y", res)
    res = check_elementwise(dx, r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert res, ("dx", res)
    res = check_reduction(np.array([dw]), np.array([r["dw"]]), np.array([r["dw_abs"]]), x.numel(),
                          GRAD_TOL)
    assert res and res.clause2 == 0, ("dw", res, dw, r["dw"])
    return res


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 100, 4095, 4096, 4097, 65539, 1_000_003])
def test_silu_parity(wsf, dt, n):
    x, dy, w = make_silu(n, dt)
    assert_silu_parity(x, dy, w, *run_silu(wsf, x, dy, w))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("misalign", [1, 3])
def test_silu_misaligned(wsf, dt, misalign):
    x, dy, w = make_silu(10007, dt, w=-1.5)
    assert_silu_parity(x, dy, w, *run_silu(wsf, x, dy, w, misalign=misalign))


def test_silu_special_values(wsf):
    x = torch.tensor([0.0, -0.0, float("nan"), 30.0, -30.0, 65504.0, -65504.0, -1.2783203125],
                     dtype=torch.float16)
    dy = torch.tensor([1.0, -2.0, 1.0, 1.0, 1.0, 1.0, 1.0, 3.0], dtype=torch.float16)
    w = torch.tensor([0.75])
    y, dx, dw = run_silu(wsf, x, dy, w)
    assert y[0] == 0 and y[1] == 0 and torch.isnan(y[2]) and torch.isnan(dx[2])
    assert float(dx[0]) == 0.375 and float(dx[1]) == -0.75  # dy·w/2 exactly
    assert math.isnan(dw)  # a NaN input reaches the sum
    keep = torch.tensor([0, 1, 3, 4, 5, 6, 7])
    yk, dxk, dwk = run_silu(wsf, x[keep], dy[keep], w)
    assert_silu_parity(x[keep], dy[keep], w, yk, dxk, dwk)


def test_silu_zero_weight_and_empty(wsf):
    x, dy, _ = make_silu(1000, "f16")
    w = torch.tensor([0.0])
    y, dx, dw = run_silu(wsf, x, dy, w)
    assert bool((y.float() == 0).all()) and bool((dx.float() == 0).all())
    assert_silu_parity(x, dy, w, y, dx, dw)
    e = torch.empty(0, dtype=torch.float16, device=DEV)
    dwt = torch.full((1,), 4.0, device=DEV)
    wsf.silu_bwd(e, e, torch.ones(1, device=DEV), dw=dwt)
    assert float(dwt) == 0.0
    dwt.fill_(4.0)
    wsf.silu_bwd(e, e, torch.ones(1, device=DEV), dw=dwt, accumulate=True)
    assert float(dwt) == 4.0


@pytest.mark.parametrize("dt", DTS)
def test_silu_bit_reproducible_and_accumulate(wsf, dt):
    x, dy, w = make_silu(1 << 20, dt)
    xd, gd, wd = x.to(DEV), dy.to(DEV), w.to(DEV)
    outs = [wsf.silu_bwd(gd, xd, wd) for _ in range(3)]
    torch.cuda.synchronize()
    for dx, dw in outs[1:]:
        assert torch.equal(dx, outs[0][0])
        assert torch.equal(dw.view(torch.int32), outs[0][1].view(torch.int32))
    acc = torch.tensor([1.25], device=DEV)
    wsf.silu_bwd(gd, xd, wd, dw=acc, accumulate=True)
    torch.cuda.synchronize()
    assert float(acc) == float(np.float32(1.25) + np.float32(float(outs[0][1])))


# ------------------------------------------------------------- workloads, reduced
@pytest.mark.parametrize("name,N", [("c1", 100), ("c3", 3001), ("c4", 100_003), ("c5", 37)])
def test_workload_recipes_reduced(wsf, name, N):
    """The weighted-sum workloads' distributions and widths at a reduced row
    count (the full sizes are checked on sampled outputs elsewhere)."""
    import inputgen
    from inputgen.workloads import WORKLOADS
    wl = WORKLOADS[name]
    x = inputgen.make((N, wl.D), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0)
    w = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1)
    dy = inputgen.make((N,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
    y, dx, gw = run_ws(wsf, x, w, dy, block_n=wl.block_n)
    assert_ws_parity(x, w, dy, y, dx, gw)


def test_silu_workload_reduced(wsf):
    import inputgen
    from inputgen.workloads import WORKLOADS
    wl = WORKLOADS["c2"]
    n = 1 << 21
    x = inputgen.make((n,), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0)
    dy = inputgen.make((n,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
    w = torch.tensor([wl.w_scalar])
    assert_silu_parity(x, dy, w, *run_silu(wsf, x, dy, w))
