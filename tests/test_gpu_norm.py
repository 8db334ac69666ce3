"""GPU parity of RMSNorm and LayerNorm, forward and backward, against the fp64
oracle: every row-width class of the staged path, the cluster path (rows of
8193..65536 elements over clusters of 3 to 16 CTAs, ragged last slices,
clusters that walk several row tiles), the element-wise path (unaligned or
wider than 65536), row strides and guard bands, constant rows,
rows with a large common offset or with massive outlier columns, tall inputs
that fill all 912 row tiles, accumulate, empty extents, bit reproducibility,
and the measurement size (sampled dx rows, full grad_w / grad_b)."""
import numpy as np
import pytest
import torch

import oracle
from inputgen import NORMAL
from tolerance import GRAD_TOL, check_elementwise, check_reduction

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTS = ["f32", "f16", "bf16"]
EPS = 2.0 ** -17  # exactly representable in binary32, so both sides use the same eps


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def _inputs(N, D, dt, seed=0, mean=0.0):
    import inputgen
    x = inputgen.make((N, D), dt, NORMAL, mean, 1.0, seed, 0)
    w = inputgen.make((D,), "f32", NORMAL, 1.0, 0.1, seed, 1)
    dy = inputgen.make((N, D), dt, NORMAL, 0.0, 1.0, seed, 2)
    b = inputgen.make((D,), "f32", NORMAL, 0.0, 0.1, seed, 3)
    return x, w, dy, b


def _place(t, ld, mis, fill=None):
    """t [N, D] copied into a device buffer with row stride ld, shifted by mis
    elements, inside guard bands; returns (buffer, view)."""
    N, D = t.shape
    buf = torch.full((N * ld + mis + 64,), 7.0 if fill is None else fill, dtype=t.dtype,
                     device=DEV)
    v = buf[mis:mis + N * ld].view(N, ld)[:, :D]
    if fill is None:
        v.copy_(t.to(DEV))
    return buf, v


def _guards_kept(buf, N, D, ld, mis):
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask[mis:mis + N * ld].view(N, ld)[:, :D] = False
    return bool((buf[mask] == 7.0).all())


def _run(wsf, layer, x, w, dy, b, pad=0, mis=0):
    N, D = x.shape
    ld = D + pad
    _, xd = _place(x, ld, mis)
    _, gd = _place(dy, ld, mis)
    yb, y = _place(x, ld, mis, fill=7.0)
    dxb, dx = _place(x, ld, mis, fill=7.0)
    wd, bd = w.to(DEV), b.to(DEV)
    if layer:
        wsf.layernorm_fwd(xd, wd, bd, EPS, y=y)
        _, gw, gb = wsf.layernorm_bwd(xd, wd, gd, EPS, dx=dx)
    else:
        wsf.rmsnorm_fwd(xd, wd, EPS, y=y)
        _, gw = wsf.rmsnorm_bwd(xd, wd, gd, EPS, dx=dx)
        gb = None
    torch.cuda.synchronize()
    assert _guards_kept(yb, N, D, ld, mis) and _guards_kept(dxb, N, D, ld, mis)
    return y.cpu(), dx.cpu(), gw.cpu(), (gb.cpu() if gb is not None else None)


def _check(layer, x, w, dy, b, y, dx, gw, gb, dx_rows=None):
    f = oracle.norm_fwd(x, w, b if layer else None, EPS, layer)
    res = check_elementwise(y, f["y"], f["y_exact"], scale=f["y_scale"])
    assert res, ("y", res)
    if not layer:
        assert res.clause2 == 0, ("y (no cancellation in RMSNorm)", res)
    r = oracle.norm_bwd(x, w, dy, EPS, layer)
    res = check_elementwise(dx, r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert res, ("dx", res)
    N = x.shape[0]
    res = check_reduction(gw, r["grad_w"], r["grad_w_abs"], N, GRAD_TOL)
    assert res, ("grad_w", res)
    if layer:
        res = check_reduction(gb, r["grad_b"], r["grad_b_abs"], N, GRAD_TOL)
        assert res, ("grad_b", res)


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(1, 1), (7, 5), (33, 64), (100, 1000), (9, 2048), (70, 4096),
                                 (3, 8192), (2, 8200), (3, 12000), (1000, 16), (130, 200)])
def test_norm_parity(wsf, layer, dt, N, D):
    x, w, dy, b = _inputs(N, D, dt)
    _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("pad,mis", [(8, 0), (3, 0), (0, 1)])
def test_norm_strides_alignment(wsf, layer, dt, pad, mis):
    x, w, dy, b = _inputs(37, 1024, dt)
    _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b, pad=pad, mis=mis))


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_norm_all_tiles(wsf, layer, dt):
    # 70,001 rows: all 912 row tiles, tiles of 76 or 77 rows, ragged groups
    x, w, dy, b = _inputs(70001, 24, dt, seed=3)
    _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("dt", DTS)
def test_norm_constant_and_offset_rows(wsf, dt):
    x, w, dy, b = _inputs(40, 512, dt, seed=5, mean=100.0)  # large common offset
    x[3] = 0.0         # RMSNorm: r = 1/sqrt(eps); LayerNorm: y = b
    x[4] = 0.25        # LayerNorm: zero variance
    x[5, ::2] = -2.0   # LayerNorm: two-valued row
    x[5, 1::2] = 2.0
    for layer in (False, True):
        _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("dt", DTS)
def test_norm_outlier_columns(wsf, dt):
    # one large value in the same columns of every row (the first element of
    # the row and one inside it), as in activations with a few massive
    # features; the row mean then sits far from most elements
    x, w, dy, b = _inputs(300, 1024, dt, seed=11)
    x[:, 0] = 500.0
    x[:, 517] = -300.0
    for layer in (False, True):
        _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
def test_norm_accumulate_reproducible_empty(wsf, layer):
    x, w, dy, b = (t.to(DEV) for t in _inputs(300, 768, "bf16", seed=9))
    eps = EPS

    def bwd(gw=None, gb=None, acc=False, xx=x, gg=dy):
        if layer:
            return wsf.layernorm_bwd(xx, w, gg, eps, grad_w=gw, grad_b=gb, accumulate=acc)
        dx, g = wsf.rmsnorm_bwd(xx, w, gg, eps, grad_w=gw, accumulate=acc)
        return dx, g, None

    runs = [bwd() for _ in range(3)]
    for r in runs[1:]:
        for a, c in zip(r, runs[0]):
            assert a is None or torch.equal(a, c)
    fw = [wsf.layernorm_fwd(x, w, b, eps) if layer else wsf.rmsnorm_fwd(x, w, eps) for _ in range(2)]
    assert torch.equal(fw[0], fw[1])
    # accumulate: old + new in one binary32 add
    old_w = torch.randn(768, device=DEV)
    old_b = torch.randn(768, device=DEV)
    _, gw, gb = bwd(gw=old_w.clone(), gb=old_b.clone() if layer else None, acc=True)
    assert torch.equal(gw, old_w + runs[0][1])
    if layer:
        assert torch.equal(gb, old_b + runs[0][2])
    # N == 0: zero gradients, or unchanged ones when accumulating
    x0 = torch.empty((0, 768), dtype=torch.bfloat16, device=DEV)
    _, g0, b0 = bwd(gw=torch.full((768,), 5.0, device=DEV),
                    gb=torch.full((768,), 5.0, device=DEV) if layer else None, xx=x0, gg=x0)
    assert bool((g0 == 0).all()) and (b0 is None or bool((b0 == 0).all()))
    _, g1, _ = bwd(gw=torch.full((768,), 5.0, device=DEV),
                   gb=torch.full((768,), 5.0, device=DEV) if layer else None, acc=True, xx=x0,
                   gg=x0)
    assert bool((g1 == 5.0).all())
    y0 = wsf.layernorm_fwd(x0, w, b, eps) if layer else wsf.rmsnorm_fwd(x0, w, eps)
    torch.cuda.synchronize()
    assert y0.shape == (0, 768)


# Cluster rows: CTAs of 4096 elements, one cluster a row.
@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(300, 8200), (200, 12288), (130, 16384), (40, 32768),
                                 (37, 36864), (20, 50000), (9, 65536), (3, 65544),
                                 (1, 20000), (2, 40000)])  # clusters with no row or one
def test_norm_cluster_rows(wsf, layer, dt, N, D):
    x, w, dy, b = _inputs(N, D, dt, seed=D % 97)
    _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
def test_norm_cluster_tile_walk(wsf, layer):
    # 63 row tiles over clusters of 9 CTAs: fewer clusters fit at once, so
    # clusters take several tiles each and stage across tile boundaries
    x, w, dy, b = _inputs(4000, 36864, "bf16", seed=4)
    _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b))


@pytest.mark.parametrize("dt", DTS)
def test_norm_cluster_offset_outliers_strides(wsf, dt):
    x, w, dy, b = _inputs(40, 20000, dt, seed=6, mean=100.0)
    x[3] = 0.0
    x[4] = 0.25
    x[5, ::2] = -2.0
    x[5, 1::2] = 2.0
    x[10:, 0] = 500.0      # outliers in the first and in the last CTA's slice
    x[10:, 17000] = -300.0
    for layer in (False, True):
        _check(layer, x, w, dy, b, *_run(wsf, layer, x, w, dy, b, pad=8))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("D", [12288, 20000, 36872])
def test_norm_cluster_block_means(wsf, dt, D):
    # blocks of 512 columns (one warp's share of a 16-bit row) with means far
    # apart, a common offset and a ragged last CTA: the per-warp shifts of
    # LayerNorm's exchange differ widely from the row mean
    # enough rows that every cluster takes several, each shifted by the mean
    # of the one before
    x, w, dy, b = _inputs(480, D, dt, seed=D % 89)
    cols = torch.arange(D)
    x = (x.double() + 20.0 * ((cols // 512) % 7 - 3).double() + 40.0).to(x.dtype)
    x[5] = x[5, 0]  # a constant row
    _check(True, x, w, dy, b, *_run(wsf, True, x, w, dy, b))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_norm_cluster_nonfinite_row_keeps_others(wsf, dt):
    # a row holding NaN or ∞ leaves the rows after it (same cluster, later
    # rows; every cluster takes several) exact: y and dx of every other row
    # match the oracle
    N, D = 400, 20000
    x, w, dy, b = _inputs(N, D, dt, seed=11, mean=3.0)
    bad = [4, 9]
    x[4, 100] = float("nan")
    x[9, 5] = float("inf")
    y, dx, _, _ = _run(wsf, True, x, w, dy, b)
    keep = [i for i in range(N) if i not in bad]
    xs, gs = x[keep], dy[keep]
    f = oracle.norm_fwd(xs, w, b, EPS, True)
    res = check_elementwise(y[keep], f["y"], f["y_exact"], scale=f["y_scale"])
    assert res, ("y", res)
    r = oracle.norm_bwd(xs, w, gs, EPS, True)
    res = check_elementwise(dx[keep], r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert res, ("dx", res)
    assert not torch.isfinite(y[4]).all() and not torch.isfinite(dx[9]).all()


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
def test_norm_cluster_accumulate_reproducible(wsf, layer):
    D = 20000
    x, w, dy, b = (t.to(DEV) for t in _inputs(500, D, "bf16", seed=9))

    def bwd(gw=None, gb=None, acc=False):
        if layer:
            return wsf.layernorm_bwd(x, w, dy, EPS, grad_w=gw, grad_b=gb, accumulate=acc)
        dx, g = wsf.rmsnorm_bwd(x, w, dy, EPS, grad_w=gw, accumulate=acc)
        return dx, g, None

    runs = [bwd() for _ in range(3)]
    for r in runs[1:]:
        for a, c in zip(r, runs[0]):
            assert a is None or torch.equal(a, c)
    fw = [wsf.layernorm_fwd(x, w, b, EPS) if layer else wsf.rmsnorm_fwd(x, w, EPS) for _ in range(2)]
    assert torch.equal(fw[0], fw[1])
    old_w, old_b = torch.randn(D, device=DEV), torch.randn(D, device=DEV)
    _, gw, gb = bwd(gw=old_w.clone(), gb=old_b.clone() if layer else None, acc=True)
    assert torch.equal(gw, old_w + runs[0][1])
    if layer:
        assert torch.equal(gb, old_b + runs[0][2])


def test_norm_cluster_no_wait_timeouts(wsf):
    # every cluster launch so far exchanged its partial sums without a wait
    # running out (the counter is per process and device)
    x, w, dy, b = _inputs(64, 30000, "bf16", seed=8)
    _run(wsf, True, x, w, dy, b)
    assert wsf.cluster_wait_timeouts() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["n1", "n2", "n3", "n4"])
def test_norm_measurement_size(wsf, name):
    import inputgen
    from inputgen.workloads import WORKLOADS
    wl = WORKLOADS[name]
    layer = wl.op == "layernorm"
    assert wl.eps == EPS
    x = inputgen.make((wl.N, wl.D), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0, pin=True)
    dy = inputgen.make((wl.N, wl.D), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2, pin=True)
    w = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1)
    b = (inputgen.make((wl.D,), "f32", wl.b.kind, wl.b.a, wl.b.b, 0, 3) if layer
         else torch.zeros(wl.D))
    xd, gd, wd, bd = x.to(DEV), dy.to(DEV), w.to(DEV), b.to(DEV)
    if layer:
        y = wsf.layernorm_fwd(xd, wd, bd, EPS)
        dx, gw, gb = wsf.layernorm_bwd(xd, wd, gd, EPS)
    else:
        y = wsf.rmsnorm_fwd(xd, wd, EPS)
        dx, gw = wsf.rmsnorm_bwd(xd, wd, gd, EPS)
        gb = None
    torch.cuda.synchronize()
    # parameter gradients over all rows
    r = oracle.norm_bwd(x, w, dy, EPS, layer, want_dx=False)
    res = check_reduction(gw.cpu(), r["grad_w"], r["grad_w_abs"], wl.N, GRAD_TOL)
    assert res, ("grad_w", res)
    if layer:
        res = check_reduction(gb.cpu(), r["grad_b"], r["grad_b_abs"], wl.N, GRAD_TOL)
        assert res, ("grad_b", res)
    # y and dx on sampled rows (first, last, 254 random)
    rows = torch.from_numpy(np.unique(np.concatenate([[0, wl.N - 1],
                                                      np.random.default_rng(0).choice(wl.N, 254)])))
    xs, gs = x[rows].contiguous(), dy[rows].contiguous()
    f = oracle.norm_fwd(xs, w, b if layer else None, EPS, layer)
    res = check_elementwise(y[rows.to(DEV)].cpu(), f["y"], f["y_exact"], scale=f["y_scale"])
    assert res, ("y", res)
    rs = oracle.norm_bwd(xs, w, gs, EPS, layer)
    res = check_elementwise(dx[rows.to(DEV)].cpu(), rs["dx"], rs["dx_exact"], scale=rs["dx_scale"])
    assert res, ("dx", res)
