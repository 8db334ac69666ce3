"""Autograd glue on the GPU: gradients through torch.autograd against the
fp64 oracle (weighted sum, scaled SiLU, RMSNorm, LayerNorm, softmax), one
gradient per forward argument (None for the flag),
accumulation into .grad across micro-batches, the library's accumulate flag,
non-contiguous inputs, leading batch dimensions, and a finite-difference
gradcheck in fp32."""
import numpy as np
import pytest
import torch

import oracle
from inputgen import NORMAL
from tolerance import GRAD_TOL, TOL, check_elementwise, check_reduction

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def ag():
    import __graft_entry__
    __graft_entry__.build()
    from backward_ws_fwd_gb300 import autograd
    return autograd


def _ws_inputs(N, D, dt, seed=0):
    import inputgen
    x = inputgen.make((N, D), dt, NORMAL, 0, 1, seed, 0)
    w = inputgen.make((D,), "f32", NORMAL, 0, D ** -0.5, seed, 1)
    dy = inputgen.make((N,), dt, NORMAL, 0, 1, seed, 2)
    return x, w, dy


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_weighted_sum_autograd_matches_oracle(ag, dt):
    x, w, dy = _ws_inputs(333, 1000, dt)
    xd = x.to(DEV).requires_grad_()
    wd = w.to(DEV).requires_grad_()
    y = ag.weighted_sum(xd, wd)
    assert y.dtype == x.dtype and y.shape == (333,)
    y.backward(dy.to(DEV))
    ye, ya, yo = oracle.ws_fwd(x, w)
    assert check_reduction(y.detach().cpu(), ye, ya, 1000, TOL[x.dtype], ref_rounded=yo)
    r = oracle.ws_bwd(x, w, dy)
    assert check_elementwise(xd.grad.cpu(), r["dx"], np.outer(dy.double(), w.double()))
    assert check_reduction(wd.grad.cpu(), r["grad_w"], r["grad_w_abs"], 333, GRAD_TOL)


def test_weighted_sum_batch_dims_and_noncontiguous(ag):
    import inputgen
    x = inputgen.make((4, 7, 64), "bf16", NORMAL, 0, 1, 0, 0)
    w = inputgen.make((64,), "f32", NORMAL, 0, 0.125, 0, 1)
    xd = x.to(DEV).transpose(0, 1).contiguous().transpose(0, 1).requires_grad_()  # strided view
    assert not xd.is_contiguous()
    wd = w.to(DEV).requires_grad_()
    y = ag.weighted_sum(xd, wd)
    assert y.shape == (4, 7)
    dy = torch.randn(4, 7, dtype=torch.bfloat16, device=DEV)
    y.backward(dy)
    ref_y = (x.float() @ w).to(torch.bfloat16)
    assert (y.detach().cpu().float() - ref_y.float()).abs().max() <= 2 ** -6 * ref_y.float().abs().max()
    r = oracle.ws_bwd(x.reshape(-1, 64).contiguous(), w, dy.cpu().reshape(-1).contiguous())
    assert check_reduction(wd.grad.cpu(), r["grad_w"], r["grad_w_abs"], 28, GRAD_TOL)
    assert xd.grad.shape == x.shape


def test_grad_accumulates_across_microbatches(ag):
    """Two backward passes add into .grad (fp32 +=): the result equals the
    fp32 sum of the two single-batch gradients, bit for bit."""
    x1, w, g1 = _ws_inputs(500, 256, "f16", seed=1)
    x2, _, g2 = _ws_inputs(500, 256, "f16", seed=2)
    wd = w.to(DEV).requires_grad_()
    ag.weighted_sum(x1.to(DEV), wd).backward(g1.to(DEV))
    first = wd.grad.clone()
    ag.weighted_sum(x2.to(DEV), wd).backward(g2.to(DEV))
    wd2 = w.to(DEV).requires_grad_()
    ag.weighted_sum(x2.to(DEV), wd2).backward(g2.to(DEV))
    assert torch.equal(wd.grad, first + wd2.grad)


def test_library_accumulate_flag_microbatches(ag):
    """The same with the library's own accumulate flag (a caller-managed
    gradient buffer): grad_w = old + batch gradient, one fp32 add."""
    import backward_ws_fwd_gb300 as wsf
    x1, w, g1 = _ws_inputs(700, 64, "bf16", seed=3)
    x2, _, g2 = _ws_inputs(700, 64, "bf16", seed=4)
    wd = w.to(DEV)
    buf = torch.zeros(64, device=DEV)
    wsf.ws_bwd(x1.to(DEV), wd, g1.to(DEV), grad_w=buf, accumulate=False)
    a = buf.clone()
    wsf.ws_bwd(x2.to(DEV), wd, g2.to(DEV), grad_w=buf, accumulate=True)
    _, b = wsf.ws_bwd(x2.to(DEV), wd, g2.to(DEV))
    assert torch.equal(buf, a + b)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_scaled_silu_autograd_matches_oracle(ag, dt):
    import inputgen
    x = inputgen.make((129, 257), dt, NORMAL, 0, 2, 0, 0)
    dy = inputgen.make((129, 257), dt, NORMAL, 0, 1, 0, 2)
    xd = x.to(DEV).requires_grad_()
    wd = torch.tensor([0.75], device=DEV, requires_grad=True)
    y = ag.scaled_silu(xd, wd, True)
    y.backward(dy.to(DEV))
    ye, yo = oracle.silu_fwd(x, 0.75)
    assert check_elementwise(y.detach().cpu(), yo, ye)
    r = oracle.silu_bwd(dy, x, 0.75)
    assert check_elementwise(xd.grad.cpu(), r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert wd.grad.shape == (1,)
    assert check_reduction(wd.grad.cpu(), np.array([r["dw"]]), np.array([r["dw_abs"]]), x.numel(),
                           GRAD_TOL)


def test_backward_returns_one_grad_per_input(ag):
    x = torch.randn(8, 16, device=DEV, requires_grad=True)
    w = torch.tensor([0.5], device=DEV, requires_grad=True)
    y = ag.ScaledSiLUFunction.apply(x, w, False)
    grads = torch.autograd.grad(y.sum(), (x, w))
    assert grads[0].shape == x.shape and grads[1].shape == w.shape
    # only x needs a gradient: w's slot is None and nothing fails
    x2 = torch.randn(8, 16, device=DEV, requires_grad=True)
    w2 = torch.tensor([0.5], device=DEV)
    (gx,) = torch.autograd.grad(ag.scaled_silu(x2, w2).sum(), (x2,))
    assert gx.shape == x2.shape


def test_modules_train_step(ag):
    """One optimizer step through both modules (a tiny regression)."""
    torch.manual_seed(0)
    ws = ag.WeightedSum(64, device=DEV)
    act = ag.ScaledSiLU(1.0, device=DEV)
    opt = torch.optim.SGD(list(ws.parameters()) + list(act.parameters()), lr=0.1)
    x = torch.randn(256, 64, device=DEV)
    target = torch.randn(256, device=DEV)
    losses = []
    for _ in range(5):
        opt.zero_grad()
        loss = ((act(ws(x).unsqueeze(1)).squeeze(1) - target) ** 2).mean()
        loss.backward()
        opt.step()
        losses.append(float(loss))
    assert losses[-1] < losses[0]


def test_gradcheck_fp32(ag):
    """Finite differences in fp32 (the kernels have no fp64 path), with
    tolerances sized for fp32 differences."""
    x = torch.randn(6, 5, device=DEV, dtype=torch.float32, requires_grad=True)
    w = torch.randn(5, device=DEV, dtype=torch.float32, requires_grad=True)
    assert torch.autograd.gradcheck(ag.weighted_sum, (x, w), eps=1e-2, atol=1e-3, rtol=1e-3,
                                    check_grad_dtypes=False, raise_exception=True)
    xs = torch.randn(7, device=DEV, dtype=torch.float32, requires_grad=True)
    ws = torch.tensor([0.8], device=DEV, requires_grad=True)
    assert torch.autograd.gradcheck(lambda a, b: ag.scaled_silu(a, b), (xs, ws), eps=1e-2,
                                    atol=2e-3, rtol=2e-3, check_grad_dtypes=False,
                                    raise_exception=True)


@pytest.mark.parametrize("layer", [False, True], ids=["rms", "ln"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_norm_autograd_matches_oracle(ag, layer, dt):
    import inputgen
    eps = 2.0 ** -17
    x = inputgen.make((3, 50, 768), dt, NORMAL, 0.2, 1, 4, 0)   # leading batch dims
    w = inputgen.make((768,), "f32", NORMAL, 1, 0.1, 4, 1)
    b = inputgen.make((768,), "f32", NORMAL, 0, 0.1, 4, 3)
    dy = inputgen.make((3, 50, 768), dt, NORMAL, 0, 1, 4, 2)
    xd = x.to(DEV).requires_grad_()
    wd = w.to(DEV).requires_grad_()
    bd = b.to(DEV).requires_grad_()
    y = ag.layer_norm(xd, wd, bd, eps) if layer else ag.rms_norm(xd, wd, eps)
    assert y.shape == x.shape and y.dtype == x.dtype
    y.backward(dy.to(DEV).transpose(0, 1).contiguous().transpose(0, 1))  # non-contiguous dy
    x2, dy2 = x.reshape(-1, 768), dy.reshape(-1, 768)
    f = oracle.norm_fwd(x2, w, b if layer else None, eps, layer)
    assert check_elementwise(y.detach().cpu().reshape(-1, 768), f["y"], f["y_exact"],
                             scale=f["y_scale"])
    r = oracle.norm_bwd(x2, w, dy2, eps, layer)
    assert check_elementwise(xd.grad.cpu().reshape(-1, 768), r["dx"], r["dx_exact"],
                             scale=r["dx_scale"])
    assert check_reduction(wd.grad.cpu(), r["grad_w"], r["grad_w_abs"], 150, GRAD_TOL)
    if layer:
        assert check_reduction(bd.grad.cpu(), r["grad_b"], r["grad_b_abs"], 150, GRAD_TOL)
    else:
        assert bd.grad is None


def test_norm_modules_accumulate_grad(ag):
    m = ag.LayerNorm(256, device=DEV)
    x = torch.randn(64, 256, device=DEV)
    g = torch.randn(64, 256, device=DEV)
    m(x).backward(g)
    first = m.weight.grad.clone(), m.bias.grad.clone()
    m(x).backward(g)  # a second micro-batch: PyTorch adds into .grad
    assert torch.equal(m.weight.grad, first[0] + first[0])
    assert torch.equal(m.bias.grad, first[1] + first[1])
    r = ag.RMSNorm(256, device=DEV)
    r(x.to(torch.bfloat16)).float().sum().backward()
    assert r.weight.grad is not None and r.weight.grad.shape == (256,)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("D", [1000, 50257])
def test_softmax_autograd_matches_oracle(ag, dt, D):
    # leading batch dimensions, a windowed width (50257) on the cluster path,
    # and a non-contiguous incoming gradient
    import inputgen
    x = inputgen.make((2, 3, D), dt, NORMAL, 0, 2, 6, 0)
    dy = inputgen.make((2, 3, D), dt, NORMAL, 0, 1, 6, 2)
    xd = x.to(DEV).requires_grad_()
    y = ag.softmax(xd)
    assert y.shape == x.shape and y.dtype == x.dtype
    y.backward(dy.to(DEV).transpose(0, 1).contiguous().transpose(0, 1))
    x2, dy2 = x.reshape(-1, D), dy.reshape(-1, D)
    ye, yo = oracle.softmax_fwd(x2)
    assert check_elementwise(y.detach().cpu().reshape(-1, D), yo, ye)
    r = oracle.softmax_bwd(y.detach().cpu().reshape(-1, D), dy2)
    assert check_elementwise(xd.grad.cpu().reshape(-1, D), r["dx"], r["dx_exact"],
                             scale=r["dx_scale"])


def test_softmax_gradcheck_fp32(ag):
    x = torch.randn(4, 9, device=DEV, dtype=torch.float32, requires_grad=True)
    assert torch.autograd.gradcheck(ag.softmax, (x,), eps=1e-2, atol=2e-3, rtol=2e-3,
                                    check_grad_dtypes=False, raise_exception=True)
