"""torch.autograd glue over the C ABI: the operators as differentiable ops.

"Writing Triton Kernels with Autograd: A Minimal End-to-End Example", §5
Wrapping with torch.autograd.Function, and "Backward in Triton —
autograd.Function and the backward grid", § A complete minimal example:
the forward saves (x, w), the backward receives dy and returns one gradient
per forward argument, in order, with None for a non-differentiable flag.
Both gradients of each operator come from one backward launch pair (stage 1
and the fixed-order stage 2); nothing here computes anything itself.

RMSNorm and LayerNorm follow "Backward in Triton — autograd.Function and
the backward grid", § Save vs recompute: the forward saves only x and the
parameters, and the backward recomputes the row statistics from x.  Softmax
saves its output y, from which its backward is formed ("Backprop for kernel
writers", §04 The duality: dx = y ⊙ (dy − Σ dy·y)).

Gradient accumulation across micro-batches ("fp32 accumulation, and why
gradients use +=") happens in PyTorch's engine, which adds each returned
gradient into ``.grad``; callers that manage gradient buffers themselves use
``accumulate=True`` of :func:`backward_ws_fwd_gb300.ws_bwd` /
:func:`backward_ws_fwd_gb300.silu_bwd` instead.
"""
from __future__ import annotations

import torch

from . import (layernorm_bwd, layernorm_fwd, rmsnorm_bwd, rmsnorm_fwd, silu_bwd, silu_fwd,
               softmax_bwd, softmax_fwd, ws_bwd, ws_fwd)

_STORAGE = (torch.float32, torch.float16, torch.bfloat16)


def _rows(x: torch.Tensor) -> torch.Tensor:
    """x as [N, D] with unit inner stride (the contiguity guard: a tensor that
    arrives non-contiguous is copied, any row stride is kept)."""
    x2 = x.reshape(-1, x.shape[-1]) if x.dim() != 2 else x
    if x2.stride(-1) != 1 or (x2.shape[0] > 1 and x2.stride(0) < x2.shape[1]):
        x2 = x2.contiguous()
    return x2


class WeightedSumFunction(torch.autograd.Function):
    """y[..., ] = Σ_d x[..., d]·w[d] for x of storage type fp32/fp16/bf16 and
    w fp32 [D]; y has x's type and x's leading shape."""

    @staticmethod
    def forward(ctx, x, w):
        if x.dtype not in _STORAGE or w.dtype != torch.float32:
            raise TypeError("x must be float32/float16/bfloat16 and w float32")
        lead = x.shape[:-1]
        x2 = _rows(x)
        w = w.contiguous()
        y = ws_fwd(x2, w)
        ctx.save_for_backward(x2, w)
        ctx.x_shape = x.shape
        return y.reshape(lead)

    @staticmethod
    def backward(ctx, dy):
        x2, w = ctx.saved_tensors
        dy = dy.reshape(-1).contiguous()  # dy can arrive non-contiguous
        dx, grad_w = ws_bwd(x2, w, dy)
        need_x, need_w = ctx.needs_input_grad
        return (dx.reshape(ctx.x_shape) if need_x else None), (grad_w if need_w else None)


class ScaledSiLUFunction(torch.autograd.Function):
    """y = w·x·sigmoid(x) with a one-element fp32 w on the device.  `inplace`
    is a non-differentiable flag kept for interface parity with the page's
    example; as there, it does not change what is computed (y is a new
    tensor, and x is saved for the backward, which recomputes sigmoid(x))."""

    @staticmethod
    def forward(ctx, x, w, inplace=False):
        if x.dtype not in _STORAGE or w.dtype != torch.float32 or w.numel() != 1:
            raise TypeError("x must be float32/float16/bfloat16 and w a one-element float32")
        x = x.contiguous()
        y = silu_fwd(x, w)
        ctx.save_for_backward(x, w)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        dy = dy.contiguous()
        dx, dw = silu_bwd(dy, x, w)
        need_x, need_w, _ = ctx.needs_input_grad
        return (dx if need_x else None), (dw.reshape(w.shape) if need_w else None), None


class RMSNormFunction(torch.autograd.Function):
    """y = x·r·w over the last dimension, r = 1/sqrt(mean x² + eps); x of
    storage type fp32/fp16/bf16 (y has x's type), w fp32 [D]."""

    @staticmethod
    def forward(ctx, x, w, eps=1e-5):
        if x.dtype not in _STORAGE or w.dtype != torch.float32:
            raise TypeError("x must be float32/float16/bfloat16 and w float32")
        x2 = _rows(x)
        w = w.contiguous()
        y = rmsnorm_fwd(x2, w, eps)
        ctx.save_for_backward(x2, w)
        ctx.eps, ctx.x_shape = eps, x.shape
        return y.reshape(x.shape)

    @staticmethod
    def backward(ctx, dy):
        x2, w = ctx.saved_tensors
        dy = _rows(dy.reshape(x2.shape))
        dx, grad_w = rmsnorm_bwd(x2, w, dy, ctx.eps)
        need_x, need_w, _ = ctx.needs_input_grad
        return (dx.reshape(ctx.x_shape) if need_x else None), (grad_w if need_w else None), None


class LayerNormFunction(torch.autograd.Function):
    """y = (x − mean)·r·w + b over the last dimension, r = 1/sqrt(var + eps)."""

    @staticmethod
    def forward(ctx, x, w, b, eps=1e-5):
        if x.dtype not in _STORAGE or w.dtype != torch.float32 or b.dtype != torch.float32:
            raise TypeError("x must be float32/float16/bfloat16, w and b float32")
        x2 = _rows(x)
        w, b = w.contiguous(), b.contiguous()
        y = layernorm_fwd(x2, w, b, eps)
        ctx.save_for_backward(x2, w)
        ctx.eps, ctx.x_shape = eps, x.shape
        return y.reshape(x.shape)

    @staticmethod
    def backward(ctx, dy):
        x2, w = ctx.saved_tensors
        dy = _rows(dy.reshape(x2.shape))
        dx, grad_w, grad_b = layernorm_bwd(x2, w, dy, ctx.eps)
        need_x, need_w, need_b, _ = ctx.needs_input_grad
        return ((dx.reshape(ctx.x_shape) if need_x else None), (grad_w if need_w else None),
                (grad_b if need_b else None), None)


class SoftmaxFunction(torch.autograd.Function):
    """Softmax over the last dimension for storage types fp32/fp16/bf16; the
    output has x's type and shape."""

    @staticmethod
    def forward(ctx, x):
        if x.dtype not in _STORAGE:
            raise TypeError("x must be float32/float16/bfloat16")
        x2 = _rows(x)
        y = softmax_fwd(x2)
        ctx.save_for_backward(y)
        ctx.x_shape = x.shape
        return y.reshape(x.shape)

    @staticmethod
    def backward(ctx, dy):
        (y,) = ctx.saved_tensors
        dy = _rows(dy.reshape(y.shape))
        return softmax_bwd(y, dy).reshape(ctx.x_shape)


def softmax(x: torch.Tensor) -> torch.Tensor:
    return SoftmaxFunction.apply(x)


def rms_norm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-5) -> torch.Tensor:
    return RMSNormFunction.apply(x, w, eps)


def layer_norm(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor, eps: float = 1e-5) -> torch.Tensor:
    return LayerNormFunction.apply(x, w, b, eps)


def weighted_sum(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    return WeightedSumFunction.apply(x, w)


def scaled_silu(x: torch.Tensor, w: torch.Tensor, inplace: bool = False) -> torch.Tensor:
    return ScaledSiLUFunction.apply(x, w, inplace)


class WeightedSum(torch.nn.Module):
    """A learnable weight vector w[D] (fp32) applied as y = x·w."""

    def __init__(self, D: int, device=None):
        super().__init__()
        self.w = torch.nn.Parameter(torch.empty(D, dtype=torch.float32, device=device))
        torch.nn.init.normal_(self.w, std=D ** -0.5)

    def forward(self, x):
        return weighted_sum(x, self.w)


class ScaledSiLU(torch.nn.Module):
    """A learnable scalar gate w (fp32) applied as y = w·silu(x)."""

    def __init__(self, init: float = 1.0, device=None):
        super().__init__()
        self.w = torch.nn.Parameter(torch.full((1,), float(init), dtype=torch.float32,
                                               device=device))

    def forward(self, x):
        return scaled_silu(x, self.w)


class RMSNorm(torch.nn.Module):
    """RMSNorm over the last dimension with a learnable fp32 scale (init 1)."""

    def __init__(self, D: int, eps: float = 1e-5, device=None):
        super().__init__()
        self.eps = eps
        self.weight = torch.nn.Parameter(torch.ones(D, dtype=torch.float32, device=device))

    def forward(self, x):
        return rms_norm(x, self.weight, self.eps)


class LayerNorm(torch.nn.Module):
    """LayerNorm over the last dimension with learnable fp32 scale and shift."""

    def __init__(self, D: int, eps: float = 1e-5, device=None):
        super().__init__()
        self.eps = eps
        self.weight = torch.nn.Parameter(torch.ones(D, dtype=torch.float32, device=device))
        self.bias = torch.nn.Parameter(torch.zeros(D, dtype=torch.float32, device=device))

    def forward(self, x):
        return layer_norm(x, self.weight, self.bias, self.eps)
