"""Pins for the oracle's weighted sum (forward and backward).

Definitions (page "Writing Triton Kernels with Autograd: A Minimal
End-to-End Example"): §1 y[i] = Σ_d x[i,d]·w[d]; §3 grad_x = dy[:,None]·w,
grad_w = Σ_i x[i,:]·dy[i], and the per-tile partial rows.  Each test pins the
oracle to something other than its own formula: the worked shape, textbook
special cases, a library GEMV, the adjoint identity that ties forward to
backward, finite differences and a materialised Jacobian, and integer inputs
whose sums are exact in any order.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from inputgen import NORMAL, UNIFORM

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _x(N, D, dt="f32", stream=0, dist=NORMAL, a=0.0, b=1.0, ig=None):
    return ig.make((N, D), dt, dist, a, b, seed=0, stream=stream)


def test_worked_shape(orc, ig):
    g = json.load(open(os.path.join(GOLD, "ws_worked_shape.json")))
    N, D, bn = g["rows"], g["d"], g["block_n"]
    x = ig.make((N, D), "f32", NORMAL, 0, 1, 0, 0)
    w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
    dy = ig.make((N,), "f32", NORMAL, 0, 1, 0, 2)
    r = orc.ws_bwd(x, w, dy, block_n=bn)
    part = r["partial"]
    assert math.ceil(N / bn) == g["n_row_tiles"]
    assert list(part.shape) == g["partial_shape"]
    assert list(r["grad_w"].shape) == g["grad_w_shape"]
    # each tile row is the sum over exactly its rows (the last tile has 4)
    for p, (a, b) in enumerate(g["tile_rows"]):
        sub = orc.ws_bwd(x[a:b + 1].contiguous(), w, dy[a:b + 1].contiguous())
        assert np.array_equal(part[p], sub["grad_w"])
    # stage 2: the sum over tiles is grad_w (to fp64 rounding)
    s = part.sum(axis=0)
    assert np.allclose(s, r["grad_w"], rtol=0, atol=1e-12 * r["grad_w_abs"].max())


def test_forward_is_a_gemv(orc, ig):
    """y equals a library fp64 matrix-vector product of the same inputs."""
    for (N, D, dt) in [(1, 1, "f32"), (7, 5, "f16"), (33, 129, "bf16"), (100, 64, "f32")]:
        x = ig.make((N, D), dt, NORMAL, 0, 1, 0, 0)
        w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
        ye, ya, _ = orc.ws_fwd(x, w)
        ref = x.double().numpy() @ w.double().numpy()
        assert np.all(np.abs(ye - ref) <= 4 * D * 2.0 ** -53 * ya)
        assert np.allclose(ya, np.abs(x.double().numpy()) @ np.abs(w.double().numpy()))


def test_grad_w_is_x_transpose_dy(orc, ig):
    for (N, D, dt) in [(1, 3, "f32"), (7, 5, "f16"), (100, 64, "f32"), (257, 17, "bf16")]:
        x = ig.make((N, D), dt, NORMAL, 0, 1, 0, 0)
        w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
        dy = ig.make((N,), dt, NORMAL, 0, 1, 0, 2)
        r = orc.ws_bwd(x, w, dy)
        ref = x.double().numpy().T @ dy.double().numpy()
        assert np.all(np.abs(r["grad_w"] - ref) <= 4 * N * 2.0 ** -53 * r["grad_w_abs"])


def test_special_cases(orc, ig):
    N, D = 7, 5
    x = ig.make((N, D), "f32", NORMAL, 0, 1, 0, 0)
    # w = e_d selects column d exactly
    for d in range(D):
        w = torch.zeros(D, dtype=torch.float32)
        w[d] = 1.0
        ye, _, yo = orc.ws_fwd(x, w)
        assert np.array_equal(ye, x[:, d].double().numpy())
        assert torch.equal(yo, x[:, d])
    # dy = e_i gives grad_w = x[i, :]
    w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
    for i in range(N):
        dy = torch.zeros(N, dtype=torch.float32)
        dy[i] = 1.0
        r = orc.ws_bwd(x, w, dy)
        assert np.array_equal(r["grad_w"], x[i].double().numpy())
        # and dx rows other than i are zero, row i is w
        assert torch.equal(r["dx"][i], w) and torch.count_nonzero(r["dx"][torch.arange(N) != i]) == 0
    # dy = 1 gives column sums
    dy = torch.ones(N, dtype=torch.float32)
    r = orc.ws_bwd(x, w, dy)
    cs = np.array([math.fsum(x[:, d].double().tolist()) for d in range(D)])
    assert np.all(np.abs(r["grad_w"] - cs) <= 4 * N * 2.0 ** -53 * r["grad_w_abs"])


def test_adjoint_identity(orc, ig):
    """<dy, y> = <w, grad_w> = <x, dx>: all three are dyᵀ·x·w.  A transposed
    operand, a dropped term or a sign error in either direction breaks it."""
    for (N, D, dt) in [(1, 64, "f32"), (7, 5, "f32"), (100, 64, "f32"), (64, 300, "f16")]:
        x = ig.make((N, D), dt, NORMAL, 0, 1, 0, 0)
        w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
        dy = ig.make((N,), dt, NORMAL, 0, 1, 0, 2)
        ye, ya, _ = orc.ws_fwd(x, w)
        r = orc.ws_bwd(x, w, dy)
        a = math.fsum((dy.double().numpy() * ye).tolist())
        b = math.fsum((w.double().numpy() * r["grad_w"]).tolist())
        scale = float(np.abs(dy.double().numpy()) @ ya)
        assert abs(a - b) <= 1e-12 * scale
        if dt == "f32":
            # dx is dy[i]·w[d] rounded to fp32; compare in exact terms
            dx_exact = np.outer(dy.double().numpy(), w.double().numpy())
            c = math.fsum((x.double().numpy() * dx_exact).ravel().tolist())
            assert abs(a - c) <= 1e-12 * scale


def test_finite_differences(orc, ig):
    """L(x, w) = Σ_i dy_i·y_i is linear in each input, so a central
    difference through the oracle's forward gives the backward's values."""
    N, D = 7, 6
    x = ig.make((N, D), "f32", NORMAL, 0, 1, 0, 0)
    w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
    dy = ig.make((N,), "f32", NORMAL, 0, 1, 0, 2)
    r = orc.ws_bwd(x, w, dy)
    dyv = dy.double().numpy()

    def L(xx, ww):
        return float(dyv @ orc.ws_fwd(xx, ww)[0])

    h = 2.0 ** -8
    for d in range(D):
        wp, wm = w.clone(), w.clone()
        wp[d] += h
        wm[d] -= h
        fd = (L(x, wp) - L(x, wm)) / (float(wp[d]) - float(wm[d]))
        assert abs(fd - r["grad_w"][d]) <= 1e-9 * (1 + abs(r["grad_w"][d]))
    for i in range(N):
        for d in range(D):
            xp, xm = x.clone(), x.clone()
            xp[i, d] += h
            xm[i, d] -= h
            fd = (L(xp, w) - L(xm, w)) / (float(xp[i, d]) - float(xm[i, d]))
            exact_dx = float(dy[i]) * float(w[d])
            assert abs(fd - exact_dx) <= 1e-9 * (1 + abs(exact_dx))
            # the oracle's dx is that product rounded once to fp32
            assert float(r["dx"][i, d]) == float(np.float32(exact_dx))


@pytest.mark.parametrize("N", [1, 7])
def test_brute_force_jacobian(orc, ig, N):
    """Materialise J_x (N × N·D) and J_w (N × D) by probing the oracle's
    forward with unit vectors, then check Jᵀ·dy against the backward.  Batch
    1 and batch 7: a missing reduction over the batch axis is invisible at 1."""
    D = 5
    rng = np.random.default_rng(N)
    x = torch.from_numpy(rng.integers(-3, 4, (N, D)).astype(np.float32))
    w = torch.from_numpy(rng.integers(-3, 4, D).astype(np.float32))
    dy = torch.from_numpy(rng.integers(-3, 4, N).astype(np.float32))
    y0 = orc.ws_fwd(x, w)[0]
    Jx = np.zeros((N, N * D))
    for j in range(N):
        for d in range(D):
            xp = x.clone()
            xp[j, d] += 1.0
            Jx[:, j * D + d] = orc.ws_fwd(xp, w)[0] - y0
    Jw = np.zeros((N, D))
    for d in range(D):
        wp = w.clone()
        wp[d] += 1.0
        Jw[:, d] = orc.ws_fwd(x, wp)[0] - y0
    r = orc.ws_bwd(x, w, dy)
    dyv = dy.double().numpy()
    assert np.array_equal(Jx.T @ dyv, r["dx"].double().numpy().ravel())
    assert np.array_equal(Jw.T @ dyv, r["grad_w"])


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,D", [(1, 1), (7, 5), (100, 64), (33, 1000)])
def test_integer_exact(orc, dt, N, D):
    """x, w, dy in {-1, 0, 1}: every sum is a small integer, exact in any
    order, so the oracle must equal integer arithmetic bit for bit."""
    rng = np.random.default_rng(N * 1000 + D)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]
    xi = rng.integers(-1, 2, (N, D))
    wi = rng.integers(-1, 2, D)
    gi = rng.integers(-1, 2, N)
    x = torch.from_numpy(xi.astype(np.float32)).to(tdt)
    w = torch.from_numpy(wi.astype(np.float32))
    dy = torch.from_numpy(gi.astype(np.float32)).to(tdt)
    ye, _, yo = orc.ws_fwd(x, w)
    assert np.array_equal(ye, (xi @ wi).astype(np.float64))
    assert torch.equal(yo.float(), torch.from_numpy((xi @ wi).astype(np.float32)))
    r = orc.ws_bwd(x, w, dy, block_n=32)
    assert np.array_equal(r["grad_w"], (xi.T @ gi).astype(np.float64))
    assert torch.equal(r["dx"].float(), torch.from_numpy(np.outer(gi, wi).astype(np.float32)))
    for p in range(r["partial"].shape[0]):
        a, b = 32 * p, min(N, 32 * p + 32)
        assert np.array_equal(r["partial"][p], (xi[a:b].T @ gi[a:b]).astype(np.float64))


def test_row_stride(orc, ig):
    """A row stride larger than D reads only the first D entries of a row."""
    N, D, ld = 9, 5, 8
    buf = torch.full((N, ld), float("nan"))
    buf[:, :D] = ig.make((N, D), "f32", NORMAL, 0, 1, 0, 0)
    xs = buf[:, :D]
    w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
    dy = ig.make((N,), "f32", NORMAL, 0, 1, 0, 2)
    a = orc.ws_fwd(xs, w)[0]
    b = orc.ws_fwd(xs.contiguous(), w)[0]
    assert np.array_equal(a, b)
    assert np.array_equal(orc.ws_bwd(xs, w, dy)["grad_w"], orc.ws_bwd(xs.contiguous(), w, dy)["grad_w"])


def test_dx_is_single_rounding_of_exact_product(orc, ig):
    """dx = dy·w rounded once: for fp32 numpy's fp32 multiply is that rounding;
    for fp16 numpy's double -> half conversion; for bf16 the generator's
    independently written rounding."""
    N, D = 64, 33
    w = ig.make((D,), "f32", NORMAL, 0, 1, 0, 1)
    for dt in ["f32", "f16", "bf16"]:
        x = ig.make((N, D), dt, NORMAL, 0, 1, 0, 0)
        dy = ig.make((N,), dt, NORMAL, 0, 1, 0, 2)
        r = orc.ws_bwd(x, w, dy)
        exact = np.outer(dy.double().numpy(), w.double().numpy())
        if dt == "f32":
            ref = np.outer(dy.numpy(), w.numpy()).astype(np.float32)
            assert np.array_equal(r["dx"].numpy(), ref)
        elif dt == "f16":
            assert np.array_equal(r["dx"].numpy(), exact.astype(np.float16))
        else:
            bits = np.array([ig.round_bf16_bits(v) for v in exact.ravel()], dtype=np.uint16)
            got = r["dx"].view(torch.int16).numpy().view(np.uint16).ravel()
            assert np.array_equal(got, bits)


def test_bf16_accumulation_illustration(orc):
    """The page's worked numerics example: 32,768 contributions of ~1e-3
    summed with a bf16 running total lose all but ~2 digits; an fp32 running
    total keeps ~7.  Uses the oracle's bf16 rounding for the bf16 total."""
    g = json.load(open(os.path.join(GOLD, "bf16_accumulation.json")))
    n, mag = g["terms"], g["magnitude"]
    rng = np.random.default_rng(0)
    terms = (mag * (1 + 0.1 * rng.standard_normal(n))).astype(np.float32)
    exact = math.fsum(terms.astype(np.float64).tolist())
    s_bf = 0.0
    for t in terms:
        s_bf = orc.bf16_to_f64(orc.f64_to_bf16(s_bf + float(orc.bf16_to_f64(orc.f64_to_bf16(t)))))
    s32 = np.float32(0.0)
    for t in terms:
        s32 = np.float32(s32 + t)
    digits_bf = -math.log10(abs(s_bf - exact) / exact)
    assert digits_bf <= g["bf16_digits_at_most"]
    # fp32 stays within the textbook recursive-summation bound
    assert abs(float(s32) - exact) <= (n - 1) * 2.0 ** -24 * float(np.abs(terms).sum())
    assert abs(float(s32) - exact) / exact < 1e-4
