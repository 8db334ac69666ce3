"""fp64 CPU oracle — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py`` cpu_baseline / ``--impl reference``) may import this
package.  The product library never loads it and shares no code with it.

The C source (``oracle.c``) states each definition and the page section it
follows.  This wrapper marshals host torch tensors (contiguous, CPU) into the
C entry points and returns fp64 results as numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, -O2, no fast-math, no
    contraction of a·b + c into fused multiply-adds, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", _SRC,
               "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None
_vp, _i64, _int, _dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = _dbl
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = _dbl
        L.orc_f64_to_f16.argtypes = [_dbl]
        L.orc_f64_to_f16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [_dbl]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_pairwise_sum.argtypes = [_vp, _i64]
        L.orc_pairwise_sum.restype = _dbl
        L.orc_set_threads.argtypes = [_int]
        L.orc_set_threads.restype = _int
        L.orc_ws_fwd.argtypes = [_vp, _i64, _vp, _i64, _i64, _int, _vp, _vp, _vp]
        L.orc_ws_fwd.restype = _int
        L.orc_ws_bwd.argtypes = [_vp, _i64, _vp, _vp, _i64, _i64, _int, _vp, _vp, _vp, _i64, _vp]
        L.orc_ws_bwd.restype = _int
        L.orc_silu_fwd.argtypes = [_vp, _dbl, _i64, _int, _vp, _vp]
        L.orc_silu_fwd.restype = _int
        L.orc_silu_bwd.argtypes = [_vp, _vp, _dbl, _i64, _int, _vp, _vp, _vp, _vp, _vp]
        L.orc_silu_bwd.restype = _int
        L.orc_softmax_fwd.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp]
        L.orc_softmax_fwd.restype = _int
        L.orc_softmax_bwd.argtypes = [_vp, _vp, _i64, _i64, _int, _vp, _vp, _vp, _vp]
        L.orc_softmax_bwd.restype = _int
        L.orc_norm_fwd.argtypes = [_vp, _i64, _vp, _vp, _dbl, _int, _i64, _i64, _int, _vp, _vp, _vp,
                                   _vp, _vp]
        L.orc_norm_fwd.restype = _int
        L.orc_norm_bwd.argtypes = [_vp, _i64, _vp, _vp, _dbl, _int, _i64, _i64, _int, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp]
        L.orc_norm_bwd.restype = _int
        _lib = L
    return _lib



def set_threads(n: int) -> int:
    """Use n host threads (n >= 1; results do not depend on n); returns the
    previous count."""
    return int(lib().orc_set_threads(int(n)))


def threads() -> int:
    n = lib().orc_set_threads(0)  # n < 1 leaves the count unchanged
    return int(n)

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.flags["C_CONTIGUOUS"]
        return ctypes.c_void_p(t.ctypes.data)
    assert t.device.type == "cpu"
    return ctypes.c_void_p(t.data_ptr())


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with {rc}")


def _dt_of(t) -> str:
    import torch
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


# ---------------------------------------------------------------- conversions
def f16_to_f64(bits: int) -> float:
    return lib().orc_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return lib().orc_bf16_to_f64(bits)


def f64_to_f16(v: float) -> int:
    return lib().orc_f64_to_f16(float(v))


def f64_to_bf16(v: float) -> int:
    return lib().orc_f64_to_bf16(float(v))


def pairwise_sum(t: np.ndarray) -> float:
    t = np.ascontiguousarray(t, dtype=np.float64)
    return lib().orc_pairwise_sum(_ptr(t), t.size)


# ---------------------------------------------------------------- weighted sum
def ws_fwd(x, w):
    """x: host tensor [N, D] (unit inner stride, any row stride), w: [D] fp32.
    Returns (y_exact fp64 [N], y_abs fp64 [N], y_out tensor [N] in x's dtype)."""
    import torch
    assert x.dim() == 2 and x.stride(1) == 1 and w.dtype == torch.float32 and w.is_contiguous()
    N, D = x.shape
    y_exact = np.empty(N, np.float64)
    y_abs = np.empty(N, np.float64)
    y_out = torch.empty(N, dtype=x.dtype)
    _check(lib().orc_ws_fwd(_ptr(x), x.stride(0) if N > 0 else D, _ptr(w), N, D,
                            DTYPE_CODE[_dt_of(x)], _ptr(y_exact), _ptr(y_abs), _ptr(y_out)),
           "ws_fwd")
    return y_exact, y_abs, y_out


def ws_bwd(x, w, dy, *, want_dx=True, block_n=0):
    """Returns dict with dx (tensor [N,D] contiguous, x's dtype) when want_dx,
    grad_w and grad_w_abs (fp64 [D]), and partial (fp64 [ceil(N/block_n), D])
    when block_n > 0."""
    import torch
    assert x.dim() == 2 and x.stride(1) == 1 and dy.dtype == x.dtype and dy.is_contiguous()
    N, D = x.shape
    out = {}
    dx = torch.empty((N, D), dtype=x.dtype) if want_dx else None
    gw = np.empty(D, np.float64)
    gwa = np.empty(D, np.float64)
    part = None
    if block_n > 0:
        part = np.empty(((N + block_n - 1) // block_n, D), np.float64)
    _check(lib().orc_ws_bwd(_ptr(x), x.stride(0) if N > 0 else D, _ptr(w), _ptr(dy), N, D,
                            DTYPE_CODE[_dt_of(x)], _ptr(dx), _ptr(gw), _ptr(gwa), block_n,
                            _ptr(part)), "ws_bwd")
    out["dx"], out["grad_w"], out["grad_w_abs"], out["partial"] = dx, gw, gwa, part
    return out


# ---------------------------------------------------------------- scaled SiLU
def silu_fwd(x, w: float):
    """x: contiguous host tensor (any shape). Returns (y_exact fp64, y_out tensor)."""
    import torch
    assert x.is_contiguous()
    n = x.numel()
    y_exact = np.empty(n, np.float64)
    y_out = torch.empty(x.shape, dtype=x.dtype)
    _check(lib().orc_silu_fwd(_ptr(x), float(w), n, DTYPE_CODE[_dt_of(x)], _ptr(y_exact),
                              _ptr(y_out)), "silu_fwd")
    return y_exact, y_out


def silu_bwd(dy, x, w: float, *, want_dx=True, want_dw=True):
    """Returns dict: dx_exact, dx_scale (fp64 [n]), dx (tensor, x's dtype),
    dw, dw_abs (floats)."""
    import torch
    assert x.is_contiguous() and dy.is_contiguous() and dy.dtype == x.dtype
    n = x.numel()
    out = {}
    dxe = np.empty(n, np.float64) if want_dx else None
    dxs = np.empty(n, np.float64) if want_dx else None
    dx = torch.empty(x.shape, dtype=x.dtype) if want_dx else None
    dw = np.zeros(1, np.float64)
    dwa = np.zeros(1, np.float64)
    _check(lib().orc_silu_bwd(_ptr(dy), _ptr(x), float(w), n, DTYPE_CODE[_dt_of(x)], _ptr(dxe),
                              _ptr(dxs), _ptr(dx), _ptr(dw) if want_dw else None,
                              _ptr(dwa) if want_dw else None), "silu_bwd")
    out.update(dx_exact=dxe, dx_scale=dxs, dx=dx, dw=float(dw[0]), dw_abs=float(dwa[0]))
    return out


# ---------------------------------------------------------------- softmax
def softmax_fwd(x):
    """x: host tensor [N, D] (unit inner stride).  Returns (y_exact fp64
    [N, D], y_out tensor [N, D] in x's dtype)."""
    import torch
    assert x.dim() == 2 and x.stride(1) == 1
    N, D = x.shape
    ye = np.empty((N, D), np.float64)
    yo = torch.empty((N, D), dtype=x.dtype)
    _check(lib().orc_softmax_fwd(_ptr(x), x.stride(0) if N > 0 else D, N, D,
                                 DTYPE_CODE[_dt_of(x)], _ptr(ye), _ptr(yo)), "softmax_fwd")
    return ye, yo


def softmax_bwd(y, dy):
    """y, dy: contiguous host tensors [N, D].  Returns dict dx_exact,
    dx_scale (fp64 [N, D]), dx (tensor), s (fp64 [N])."""
    import torch
    assert y.is_contiguous() and dy.is_contiguous() and y.dtype == dy.dtype
    N, D = y.shape
    dxe = np.empty((N, D), np.float64)
    dxs = np.empty((N, D), np.float64)
    dx = torch.empty((N, D), dtype=y.dtype)
    s = np.empty(N, np.float64)
    _check(lib().orc_softmax_bwd(_ptr(y), _ptr(dy), N, D, DTYPE_CODE[_dt_of(y)], _ptr(dxe),
                                 _ptr(dxs), _ptr(dx), _ptr(s)), "softmax_bwd")
    return {"dx_exact": dxe, "dx_scale": dxs, "dx": dx, "s": s}


# ---------------------------------------------------------------- RMSNorm / LayerNorm
def norm_fwd(x, w, b=None, eps=1e-5, layer=False):
    """RMSNorm (layer=False) or LayerNorm (layer=True) of the rows of x [N, D].
    Returns dict y_exact, y_scale (fp64 [N, D]), y (tensor, x's dtype), r, mu (fp64 [N])."""
    import torch
    assert x.dim() == 2 and x.stride(1) == 1 and w.dtype == torch.float32 and w.is_contiguous()
    N, D = x.shape
    ye = np.empty((N, D), np.float64)
    ys = np.empty((N, D), np.float64)
    yo = torch.empty((N, D), dtype=x.dtype)
    r = np.empty(N, np.float64)
    mu = np.empty(N, np.float64)
    _check(lib().orc_norm_fwd(_ptr(x), x.stride(0) if N > 0 else D, _ptr(w),
                              _ptr(b) if b is not None else None, float(eps), int(layer), N, D,
                              DTYPE_CODE[_dt_of(x)], _ptr(ye), _ptr(ys), _ptr(yo), _ptr(r),
                              _ptr(mu)), "norm_fwd")
    return {"y_exact": ye, "y_scale": ys, "y": yo, "r": r, "mu": mu}


def norm_bwd(x, w, dy, eps=1e-5, layer=False, *, want_dx=True):
    """Returns dict dx_exact, dx_scale (fp64 [N, D]), dx (tensor), grad_w,
    grad_w_abs, grad_b, grad_b_abs (fp64 [D]; the b ones for LayerNorm)."""
    import torch
    assert x.dim() == 2 and x.stride(1) == 1 and dy.is_contiguous() and dy.dtype == x.dtype
    N, D = x.shape
    dxe = np.empty((N, D), np.float64) if want_dx else None
    dxs = np.empty((N, D), np.float64) if want_dx else None
    dx = torch.empty((N, D), dtype=x.dtype) if want_dx else None
    gw, gwa, gb, gba = (np.zeros(D, np.float64) for _ in range(4))
    _check(lib().orc_norm_bwd(_ptr(x), x.stride(0) if N > 0 else D, _ptr(w), _ptr(dy), float(eps),
                              int(layer), N, D, DTYPE_CODE[_dt_of(x)], _ptr(dxe), _ptr(dxs),
                              _ptr(dx), _ptr(gw), _ptr(gwa), _ptr(gb), _ptr(gba)), "norm_bwd")
    return {"dx_exact": dxe, "dx_scale": dxs, "dx": dx, "grad_w": gw, "grad_w_abs": gwa,
            "grad_b": gb, "grad_b_abs": gba}
