"""Pins for the oracle's scaled SiLU (forward and backward).

Definitions (page "Backward in Triton — autograd.Function and the backward
grid", § A complete minimal example — fused scaled-SiLU): s = sigmoid(x),
y = w·x·s, dy/dx = w·(s + x·s·(1 − s)), dx = dy·dy/dx, dw = Σ dy·x·s.
Pinned by exact special cases, the sigmoid's symmetry and limits, a library
sigmoid, central finite differences through the oracle's forward, and the
identity w·dw = Σ dy·y that ties the backward's dw to the forward.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from inputgen import NORMAL


def _t(vals, dt="f32"):
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]
    return torch.tensor(vals, dtype=torch.float64).to(tdt)


def test_zero_input(orc):
    """x = 0: s = 1/2, so y = 0, dx = dy·w/2 exactly, and no dw contribution."""
    x = _t([0.0, 0.0, 0.0])
    dy = _t([1.0, -3.0, 0.5])
    w = 0.75
    ye, yo = orc.silu_fwd(x, w)
    assert np.all(ye == 0.0) and torch.all(yo == 0)
    r = orc.silu_bwd(dy, x, w)
    assert np.array_equal(r["dx_exact"], dy.double().numpy() * w / 2)
    assert r["dw"] == 0.0


def test_sigmoid_matches_library(orc, ig):
    x = ig.make((4096,), "f32", NORMAL, 0.0, 4.0, 0, 0)
    x[x == 0] = 1.0
    w = 1.0
    ye, _ = orc.silu_fwd(x, w)
    s = ye / x.double().numpy()
    ref = scipy.special.expit(x.double().numpy())
    assert np.allclose(s, ref, rtol=4e-16, atol=0)


def test_odd_part_identity(orc, ig):
    """s(−x) = 1 − s(x) gives y(x) − y(−x) = w·x."""
    x = ig.make((2048,), "f32", NORMAL, 0.0, 3.0, 0, 0)
    w = -1.25
    yp, _ = orc.silu_fwd(x, w)
    ym, _ = orc.silu_fwd(-x, w)
    assert np.allclose(yp - ym, w * x.double().numpy(), rtol=1e-14, atol=1e-300)


def test_derivative_limits(orc):
    """silu'(x) → 1 as x → +∞ and → 0 as x → −∞; at the minimum of silu
    (x0 = −1 − W(1/e), where 1 + x + e^x = 0) the derivative vanishes."""
    w = 2.0
    x = _t([40.0, 80.0, -40.0, -80.0])
    dy = _t([1.0, 1.0, 1.0, 1.0])
    r = orc.silu_bwd(dy, x, w)
    assert abs(r["dx_exact"][0] - w) < 1e-15 and abs(r["dx_exact"][1] - w) < 1e-15
    assert abs(r["dx_exact"][2]) < 1e-15 and abs(r["dx_exact"][3]) < 1e-30
    x0 = -1.0 - float(scipy.special.lambertw(1.0 / math.e).real)
    xs = torch.tensor([x0], dtype=torch.float64).float()
    rr = orc.silu_bwd(_t([1.0]), xs, 1.0)
    # |silu'(x)| ≈ |x − x0| near the root (the slope there is 1)
    assert abs(rr["dx_exact"][0]) <= 2 * abs(float(xs[0]) - x0) + 1e-15


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_finite_differences_dx(orc, ig, dt):
    """dx_k = dy_k · d y_k / d x_k: central difference of the oracle's forward
    at fp32 points x ± h with a Richardson step to cancel the h² term.  The
    points sit on a 2^-12 grid and h is 2^-9 or 2^-10, so every x ± h is
    exact in fp32."""
    n = 512
    x = ig.make((n,), dt, NORMAL, 0.0, 2.0, 0, 0)
    if dt == "f32":
        x = torch.round(x * 4096) / 4096
    dy = ig.make((n,), dt, NORMAL, 0.0, 1.0, 0, 2)
    w = 0.75
    r = orc.silu_bwd(dy, x, w)
    xf = x.float()

    def diff(h):
        xp, xm = (xf + h).contiguous(), (xf - h).contiguous()
        assert torch.equal(xp.double() - xf.double(), torch.full_like(xf.double(), h))
        assert torch.equal(xf.double() - xm.double(), torch.full_like(xf.double(), h))
        yp, _ = orc.silu_fwd(xp, w)
        ym, _ = orc.silu_fwd(xm, w)
        return (yp - ym) / (2 * h)

    d1, d2 = diff(2.0 ** -9), diff(2.0 ** -10)
    fd = (4 * d2 - d1) / 3
    dyv = dy.double().numpy()
    assert np.all(np.abs(dyv * fd - r["dx_exact"]) <= 1e-9 * (r["dx_scale"] + 1e-30))


def test_dw_by_finite_difference_in_w(orc, ig):
    """y is linear in w, so (L(w+h) − L(w−h)) / 2h with L = Σ dy·y is exactly
    dL/dw = dw (up to rounding)."""
    n = 10007
    x = ig.make((n,), "f16", NORMAL, 0.0, 2.0, 0, 0)
    dy = ig.make((n,), "f16", NORMAL, 0.0, 1.0, 0, 2)
    w, h = 0.75, 0.125
    dyv = dy.double().numpy()

    def L(ww):
        return math.fsum((dyv * orc.silu_fwd(x, ww)[0]).tolist())

    fd = (L(w + h) - L(w - h)) / (2 * h)
    r = orc.silu_bwd(dy, x, w)
    assert abs(fd - r["dw"]) <= 1e-12 * r["dw_abs"]


@pytest.mark.parametrize("n", [1, 7, 4096])
def test_cross_op_identity(orc, ig, n):
    """w·dw = Σ dy·y: the backward's scalar reduction against the forward."""
    x = ig.make((n,), "bf16", NORMAL, 0.0, 2.0, 0, 0)
    dy = ig.make((n,), "bf16", NORMAL, 0.0, 1.0, 0, 2)
    w = -0.6
    ye, _ = orc.silu_fwd(x, w)
    r = orc.silu_bwd(dy, x, w)
    a = w * r["dw"]
    b = math.fsum((dy.double().numpy() * ye).tolist())
    assert abs(a - b) <= 1e-13 * abs(w) * r["dw_abs"]


def test_outputs_rounded_once(orc, ig):
    """y_out / dx_out are the fp64 values rounded once to the storage type."""
    x = ig.make((3000,), "f16", NORMAL, 0.0, 2.0, 0, 0)
    dy = ig.make((3000,), "f16", NORMAL, 0.0, 1.0, 0, 2)
    ye, yo = orc.silu_fwd(x, 0.75)
    assert np.array_equal(yo.numpy(), ye.astype(np.float16))
    r = orc.silu_bwd(dy, x, 0.75)
    assert np.array_equal(r["dx"].numpy(), r["dx_exact"].astype(np.float16))
