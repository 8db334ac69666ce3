"""Pins for the oracle's softmax and its backward ("Backprop for kernel
writers", §04: the backward is the row-scalar collapse dx = y ⊙ (dy − Σ dy·y),
expressed in terms of the output y).  Pinned by a library softmax, the
rows-sum-to-one and shift-invariance properties, the dense Jacobian
diag(y) − y·yᵀ materialised for tiny rows, finite differences through the
forward, and the invariant Σ_j dx_j = 0."""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from inputgen import NORMAL


def _x(N, D, dt="f32", sd=2.0, seed=0):
    import inputgen
    return inputgen.make((N, D), dt, NORMAL, 0.0, sd, seed, 0)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_forward_matches_library_and_sums_to_one(dt):
    x = _x(9, 257, dt)
    ye, yo = oracle.softmax_fwd(x)
    ref = scipy.special.softmax(x.double().numpy(), axis=1)
    assert np.allclose(ye, ref, rtol=1e-13, atol=0)
    assert np.allclose(ye.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert torch.equal(yo, torch.from_numpy(ye).to(x.dtype)) or dt == "bf16"


def test_shift_invariance_and_uniform():
    x = torch.round(_x(5, 64) * 4096) / 4096  # on a 2^-12 grid: x + 3 is exact in fp32
    y1, _ = oracle.softmax_fwd(x)
    y2, _ = oracle.softmax_fwd((x + 3.0).contiguous())
    assert torch.equal((x + 3.0) - 3.0, x)
    assert np.allclose(y1, y2, rtol=1e-12, atol=0)
    u, _ = oracle.softmax_fwd(torch.full((3, 10), 0.7))
    assert np.allclose(u, 0.1, rtol=0, atol=1e-16)
    # a huge entry: no overflow thanks to the max shift
    big = torch.tensor([[1000.0, 0.0, -1000.0]])
    yb, _ = oracle.softmax_fwd(big)
    assert yb[0, 0] == 1.0 and yb[0, 2] == 0.0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_masked_logits_equal_softmax_of_kept_columns(dt):
    # −inf entries (a mask) get probability exactly 0, and the kept columns
    # get the softmax of the kept sub-row; the backward is 0 where y is 0
    x = _x(4, 300, dt, seed=5)
    keep = [300, 150, 1, 77]
    xm = x.clone()
    for i, t in enumerate(keep):
        xm[i, t:] = float("-inf")
    ye, _ = oracle.softmax_fwd(xm)
    for i, t in enumerate(keep):
        ref = scipy.special.softmax(x[i, :t].double().numpy())
        assert np.allclose(ye[i, :t], ref, rtol=1e-13, atol=0)
        assert np.all(ye[i, t:] == 0.0)
    dy = _x(4, 300, dt, seed=6)
    r = oracle.softmax_bwd(torch.from_numpy(ye).to(x.dtype), dy)
    for i, t in enumerate(keep):
        assert np.all(r["dx_exact"][i, t:] == 0.0)


@pytest.mark.parametrize("D", [1, 2, 5])
def test_backward_equals_dense_jacobian(D):
    """Materialise J = diag(y) − y·yᵀ (only for the test) and compare Jᵀ·dy."""
    x = _x(4, D, "f32")
    _, yo = oracle.softmax_fwd(x)
    dy = _x(4, D, "f32", sd=1.0, seed=7)
    r = oracle.softmax_bwd(yo, dy)
    yv = yo.double().numpy()
    for i in range(4):
        J = np.diag(yv[i]) - np.outer(yv[i], yv[i])
        assert np.allclose(J.T @ dy[i].double().numpy(), r["dx_exact"][i], rtol=1e-13, atol=1e-16)


def test_backward_by_finite_differences():
    """L(x) = Σ dy·softmax(x): central differences through the oracle's
    forward equal the backward evaluated at y = softmax(x) (fp64 y)."""
    x = torch.round(_x(3, 6, "f32") * 4096) / 4096
    dy = _x(3, 6, "f32", sd=1.0, seed=3)
    ye, _ = oracle.softmax_fwd(x)
    # backward at the exact forward output, via an fp32 y close to it
    h = 2.0 ** -10
    fd = np.zeros((3, 6))
    for j in range(6):
        xp, xm = x.clone(), x.clone()
        xp[:, j] += h
        xm[:, j] -= h
        yp, _ = oracle.softmax_fwd(xp)
        ym, _ = oracle.softmax_fwd(xm)
        fd[:, j] = ((yp - ym) * dy.double().numpy()).sum(axis=1) / (2 * h)
    s = (dy.double().numpy() * ye).sum(axis=1, keepdims=True)
    exact = ye * (dy.double().numpy() - s)
    assert np.allclose(fd, exact, rtol=0, atol=1e-6)
    # and the oracle's backward on an fp32-stored y is within fp32 rounding of it
    r = oracle.softmax_bwd(torch.from_numpy(ye).float(), dy)
    assert np.allclose(r["dx_exact"], exact, rtol=0, atol=1e-6)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_backward_invariants(dt):
    x = _x(6, 300, dt)
    _, yo = oracle.softmax_fwd(x)
    dy = _x(6, 300, dt, sd=1.0, seed=5)
    r = oracle.softmax_bwd(yo, dy)
    # Σ_j dx_j = Σ_j y_j dy_j − s Σ_j y_j = s (1 − Σ y); Σ y = 1 up to the storage rounding of y
    ysum = yo.double().numpy().sum(axis=1)
    assert np.allclose(r["dx_exact"].sum(axis=1), r["s"] * (1 - ysum), rtol=1e-9, atol=1e-14)
    # a constant upstream gradient gives dx = c·y·(1 − Σ y), zero for an exactly normalised y
    c = torch.full((6, 300), 0.5, dtype=yo.dtype)
    rc = oracle.softmax_bwd(yo, c)
    assert np.allclose(rc["dx_exact"], 0.5 * yo.double().numpy() * (1 - ysum)[:, None],
                       rtol=1e-9, atol=1e-15)
