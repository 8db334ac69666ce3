"""Pins for the oracle's RMSNorm and LayerNorm (forward and backward).

The pages name both operators and their backward structure (row statistics
recomputed from x; parameter gradients reduced over the batch axis) but print
no formulas, so the oracle writes out the textbook definitions.  Pinned by
PyTorch's fp64 rms_norm / layer_norm with autograd (a library routine of the
same definition), central differences through the oracle's own forward, the
invariants that hold at eps = 0 (RMSNorm is scale-invariant: Σ_j dx_j·x_j = 0;
LayerNorm is also shift-invariant: Σ_j dx_j = 0), and a one-hot upstream
gradient, at batch 1 and batch 7."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _inputs(N, D, dt="f32", seed=0):
    g = torch.Generator().manual_seed(seed)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]
    x = (torch.randn(N, D, generator=g) * 1.5 + 0.3).to(tdt)
    w = torch.randn(D, generator=g).float()
    b = torch.randn(D, generator=g).float()
    dy = torch.randn(N, D, generator=g).to(tdt)
    return x, w, b, dy


def _torch_ref(x, w, b, dy, eps, layer):
    xd = x.double().requires_grad_()
    wd = w.double().requires_grad_()
    bd = b.double().requires_grad_()
    if layer:
        y = F.layer_norm(xd, (x.shape[1],), wd, bd, eps)
    else:
        y = F.rms_norm(xd, (x.shape[1],), wd, eps)
    y.backward(dy.double())
    return y.detach().numpy(), xd.grad.numpy(), wd.grad.numpy(), (bd.grad.numpy() if layer else None)


@pytest.mark.parametrize("layer", [False, True])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,D", [(1, 7), (7, 64), (33, 300)])
def test_matches_torch_fp64(layer, dt, N, D):
    x, w, b, dy = _inputs(N, D, dt)
    eps = 1e-5
    f = oracle.norm_fwd(x, w, b, eps, layer)
    g = oracle.norm_bwd(x, w, dy, eps, layer)
    y, dx, dw, db = _torch_ref(x, w, b, dy, eps, layer)
    assert np.allclose(f["y_exact"], y, rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dx_exact"], dx, rtol=1e-10, atol=1e-11)
    assert np.allclose(g["grad_w"], dw, rtol=1e-11, atol=1e-11)
    if layer:
        assert np.allclose(g["grad_b"], db, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("layer", [False, True])
def test_finite_differences(layer):
    x, w, b, dy = _inputs(3, 9, "f32", seed=4)
    x = torch.round(x * 1024) / 1024  # grid values: x ± h exact in fp32
    eps = 1e-3
    g = oracle.norm_bwd(x, w, dy, eps, layer)
    dyv = dy.double().numpy()

    def L(xx, ww):
        return float((oracle.norm_fwd(xx, ww, b, eps, layer)["y_exact"] * dyv).sum())

    h = 2.0 ** -9
    for i, j in [(0, 0), (1, 4), (2, 8)]:
        xp, xm = x.clone(), x.clone()
        xp[i, j] += h
        xm[i, j] -= h
        fd = (L(xp, w) - L(xm, w)) / (2 * h)
        assert abs(fd - g["dx_exact"][i, j]) <= 1e-4 * (1 + abs(fd))
    for j in [0, 5, 8]:
        wp, wm = w.clone(), w.clone()
        wp[j] += h
        wm[j] -= h
        fd = (L(x, wp) - L(x, wm)) / (float(wp[j]) - float(wm[j]))
        assert abs(fd - g["grad_w"][j]) <= 1e-8 * (1 + abs(fd))  # y is linear in w


@pytest.mark.parametrize("N", [1, 7])
def test_invariants_at_eps_zero(N):
    x, w, b, dy = _inputs(N, 50, "f32", seed=9)
    xv = x.double().numpy()
    r = oracle.norm_bwd(x, w, dy, 0.0, False)
    assert np.allclose((r["dx_exact"] * xv).sum(axis=1), 0.0, atol=1e-11)
    q = oracle.norm_bwd(x, w, dy, 0.0, True)
    assert np.allclose(q["dx_exact"].sum(axis=1), 0.0, atol=1e-11)
    assert np.allclose((q["dx_exact"] * xv).sum(axis=1), 0.0, atol=1e-10)
    # db is the column sum of dy
    assert np.allclose(q["grad_b"], dy.double().numpy().sum(axis=0), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("layer", [False, True])
def test_one_hot_upstream_gradient(layer):
    """dy = 1 on row i only: grad_w is that row's normalised values."""
    x, w, b, _ = _inputs(7, 16, "f32", seed=2)
    f = oracle.norm_fwd(x, w, b, 1e-5, layer)
    for i in [0, 3, 6]:
        dy = torch.zeros(7, 16)
        dy[i] = 1.0
        g = oracle.norm_bwd(x, w, dy, 1e-5, layer)
        xh = (x[i].double().numpy() - f["mu"][i]) * f["r"][i]
        assert np.allclose(g["grad_w"], xh, rtol=1e-14, atol=1e-15)
