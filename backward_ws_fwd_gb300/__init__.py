"""backward_ws_fwd_gb300 — Python binding of libwsfwd (C ABI in include/wsf.h).

Forward and backward (vector-Jacobian product) kernels of two memory-bound
row operators on one GB300 GPU:

* weighted sum  y[i] = Σ_d x[i,d]·w[d]   ("Writing Triton Kernels with
  Autograd: A Minimal End-to-End Example", §1–§5)
* scaled SiLU   y = w·x·sigmoid(x)        ("Backward in Triton —
  autograd.Function and the backward grid", § A complete minimal example)

This module only marshals torch tensors into the C entry points: pointers,
sizes, the storage-type code and the current CUDA stream.  Every step runs
in the library's kernels; there is no fallback.  Importing the module fails
if the library has not been built (``python -m backward_ws_fwd_gb300.build``
or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwsfwd.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libwsfwd.so is not built ({LIB_PATH}); run backward_ws_fwd_gb300/build.py")

lib = ctypes.CDLL(LIB_PATH)

_vp, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
lib.wsf_status_string.argtypes = [_int]
lib.wsf_status_string.restype = ctypes.c_char_p
lib.wsf_version.argtypes = []
lib.wsf_version.restype = _int
lib.wsf_cluster_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint), _int]
lib.wsf_cluster_wait_timeouts.restype = _int
lib.wsf_selftest_exchange_timeout.argtypes = [_vp, ctypes.c_uint, _vp]
lib.wsf_selftest_exchange_timeout.restype = _int
lib.wsf_selftest_waiting_warps.argtypes = []
lib.wsf_selftest_waiting_warps.restype = _int
lib.ws_fwd.argtypes = [_vp, _i64, _vp, _vp, _i64, _i64, _int, _vp]
lib.ws_fwd.restype = _int
lib.ws_bwd_workspace_bytes.argtypes = [_i64, _i64, _int, _i64]
lib.ws_bwd_workspace_bytes.restype = _sz
lib.ws_bwd.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _int, _vp, _sz, _i64, _i64, _i64,
                       _int, _vp]
lib.ws_bwd.restype = _int
lib.ws_bwd_noalloc.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _int, _i64, _i64, _i64, _int,
                               _vp]
lib.ws_bwd_noalloc.restype = _int
lib.ws_bwd_atomic.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _int, _i64, _i64, _int, _vp]
lib.ws_bwd_atomic.restype = _int
lib.silu_bwd_atomic.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _i64, _int, _vp]
lib.silu_bwd_atomic.restype = _int
lib.softmax_fwd.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _int, _vp]
lib.softmax_fwd.restype = _int
lib.softmax_bwd.argtypes = [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _int, _vp]
lib.softmax_bwd.restype = _int
_f = ctypes.c_float
lib.rmsnorm_fwd.argtypes = [_vp, _i64, _vp, _f, _vp, _i64, _i64, _i64, _int, _vp]
lib.rmsnorm_fwd.restype = _int
lib.layernorm_fwd.argtypes = [_vp, _i64, _vp, _vp, _f, _vp, _i64, _i64, _i64, _int, _vp]
lib.layernorm_fwd.restype = _int
lib.rmsnorm_bwd_workspace_bytes.argtypes = [_i64, _i64, _int]
lib.rmsnorm_bwd_workspace_bytes.restype = _sz
lib.layernorm_bwd_workspace_bytes.argtypes = [_i64, _i64, _int]
lib.layernorm_bwd_workspace_bytes.restype = _sz
lib.rmsnorm_bwd.argtypes = [_vp, _i64, _vp, _vp, _i64, _f, _vp, _i64, _vp, _int, _vp, _sz, _i64,
                            _i64, _int, _vp]
lib.rmsnorm_bwd.restype = _int
lib.layernorm_bwd.argtypes = [_vp, _i64, _vp, _vp, _i64, _f, _vp, _i64, _vp, _vp, _int, _vp, _sz,
                              _i64, _i64, _int, _vp]
lib.layernorm_bwd.restype = _int
lib.silu_fwd.argtypes = [_vp, _vp, _vp, _i64, _int, _vp]
lib.silu_fwd.restype = _int
lib.silu_bwd_workspace_bytes.argtypes = [_i64, _int]
lib.silu_bwd_workspace_bytes.restype = _sz
lib.silu_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _vp, _sz, _i64, _int, _vp]
lib.silu_bwd.restype = _int

F32, F16, BF16 = 0, 1, 2
SIZE_MAX = ctypes.c_size_t(-1).value

# status codes (include/wsf.h)
OK, ERR_NULL_PTR, ERR_BAD_SHAPE, ERR_BAD_DTYPE, ERR_BAD_STRIDE = 0, -1, -2, -3, -4
ERR_WORKSPACE, ERR_OVERLAP, ERR_MISALIGNED, ERR_BAD_ARG, ERR_CUDA = -5, -6, -7, -8, -9


class WsfError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def status_string(status: int) -> str:
    return lib.wsf_status_string(status).decode()


def _dtype_code(t) -> int:
    import torch
    try:
        return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported storage type {t.dtype}") from None


def _stream(stream, device=None):
    """The CUDA stream to launch on: `stream`, else the current stream of
    `device` (the tensors' device)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _on(t):
    """Make the device of tensor t current for the call: the C entry points
    launch on the current device (and ws_bwd_noalloc picks that device's
    scratch array)."""
    import contextlib
    import torch
    if t is not None and t.is_cuda:
        return torch.cuda.device(t.device)
    return contextlib.nullcontext()


def _scratch(nbytes, device, stream):
    """A temporary workspace.  It is freed when the call returns, while the
    kernels may still use it on `stream`: record that use, so the caching
    allocator does not hand the memory out before `stream` reaches this
    point (allocations on the device's current stream need nothing)."""
    import torch
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if stream is not None:
        t.record_stream(stream)
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else None


def _check(rc: int, what: str):
    if rc != OK:
        raise WsfError(rc, what)


def ws_bwd_workspace_bytes(N: int, D: int, dtype, block_n: int = 0) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code_of_dtype(dtype)
    return lib.ws_bwd_workspace_bytes(N, D, code, block_n)


def silu_bwd_workspace_bytes(n: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code_of_dtype(dtype)
    return lib.silu_bwd_workspace_bytes(n, code)


def _dtype_code_of_dtype(dt) -> int:
    import torch
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[dt]


def ws_fwd(x, w, y=None, stream=None):
    """y[i] = Σ_d x[i,d]·w[d].  x: [N, D] CUDA tensor with unit inner stride;
    w: [D] float32; y: [N] of x's dtype (allocated when None)."""
    import torch
    N, D = x.shape
    if y is None:
        y = torch.empty(N, dtype=x.dtype, device=x.device)
    with _on(x):
        _check(lib.ws_fwd(_ptr(x), x.stride(0), _ptr(w), _ptr(y), N, D, _dtype_code(x),
                          _stream(stream, x.device)), "ws_fwd")
    return y


def ws_bwd(x, w, dy, dx=None, grad_w=None, accumulate=False, workspace=None, block_n=0,
           stream=None):
    """dx[i,d] = dy[i]·w[d]; grad_w[d] (+)= Σ_i x[i,d]·dy[i].  Returns (dx, grad_w)."""
    import torch
    N, D = x.shape
    code = _dtype_code(x)
    if dx is None:
        dx = torch.empty((N, D), dtype=x.dtype, device=x.device)
    if grad_w is None:
        grad_w = torch.empty(D, dtype=torch.float32, device=x.device)
    need = lib.ws_bwd_workspace_bytes(N, D, code, block_n)
    with _on(x):
        if workspace is None and need not in (0, SIZE_MAX):
            workspace = _scratch(need, x.device, stream)
        wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib.ws_bwd(_ptr(x), x.stride(0), _ptr(w), _ptr(dy), _ptr(dx), dx.stride(0),
                          _ptr(grad_w), int(bool(accumulate)), _ptr(workspace), wbytes, block_n,
                          N, D, code, _stream(stream, x.device)), "ws_bwd")
    return dx, grad_w


def ws_bwd_noalloc(x, w, dy, dx=None, grad_w=None, accumulate=False, block_n=0, stream=None):
    """ws_bwd without a workspace argument, for callers that cannot allocate
    device memory: the partials use the library's fixed 8 MiB scratch array
    on x's device (sizes that need more are rejected).  dx and grad_w must be
    supplied by such callers; they are allocated here only for convenience
    when None."""
    import torch
    N, D = x.shape
    if dx is None:
        dx = torch.empty((N, D), dtype=x.dtype, device=x.device)
    if grad_w is None:
        grad_w = torch.empty(D, dtype=torch.float32, device=x.device)
    with _on(x):
        _check(lib.ws_bwd_noalloc(_ptr(x), x.stride(0), _ptr(w), _ptr(dy), _ptr(dx),
                                  dx.stride(0), _ptr(grad_w), int(bool(accumulate)), block_n, N,
                                  D, _dtype_code(x), _stream(stream, x.device)), "ws_bwd_noalloc")
    return dx, grad_w


def ws_bwd_atomic(x, w, dy, dx=None, grad_w=None, accumulate=False, stream=None):
    """ws_bwd with grad_w summed by atomic additions (run-to-run bits may
    differ); the measured comparison for the deterministic two-pass form."""
    import torch
    N, D = x.shape
    if dx is None:
        dx = torch.empty((N, D), dtype=x.dtype, device=x.device)
    if grad_w is None:
        grad_w = torch.empty(D, dtype=torch.float32, device=x.device)
    with _on(x):
        _check(lib.ws_bwd_atomic(_ptr(x), x.stride(0), _ptr(w), _ptr(dy), _ptr(dx), dx.stride(0),
                                 _ptr(grad_w), int(bool(accumulate)), N, D, _dtype_code(x),
                                 _stream(stream, x.device)), "ws_bwd_atomic")
    return dx, grad_w


def silu_bwd_atomic(dy, x, w, dx=None, dw=None, accumulate=False, stream=None):
    """silu_bwd with dw summed by one atomic addition per block (the pages'
    own scheme); run-to-run bits may differ."""
    import torch
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(1, dtype=torch.float32, device=x.device)
    with _on(x):
        _check(lib.silu_bwd_atomic(_ptr(dy), _ptr(x), _ptr(w), _ptr(dx),
                                   ctypes.c_void_p(dw.data_ptr()), int(bool(accumulate)),
                                   x.numel(), _dtype_code(x), _stream(stream, x.device)),
               "silu_bwd_atomic")
    return dx, dw


def softmax_fwd(x, y=None, stream=None):
    """Row softmax of x [N, D] (unit inner stride); y has x's type."""
    import torch
    N, D = x.shape
    if y is None:
        y = torch.empty((N, D), dtype=x.dtype, device=x.device)
    with _on(x):
        _check(lib.softmax_fwd(_ptr(x), x.stride(0), _ptr(y), y.stride(0), N, D, _dtype_code(x),
                               _stream(stream, x.device)), "softmax_fwd")
    return y


def softmax_bwd(y, dy, dx=None, stream=None):
    """dx = y ⊙ (dy − Σ_j dy·y) per row, from the forward's output y."""
    import torch
    N, D = y.shape
    if dx is None:
        dx = torch.empty((N, D), dtype=y.dtype, device=y.device)
    with _on(y):
        _check(lib.softmax_bwd(_ptr(y), y.stride(0), _ptr(dy), dy.stride(0), _ptr(dx),
                               dx.stride(0), N, D, _dtype_code(y), _stream(stream, y.device)),
               "softmax_bwd")
    return dx


def silu_fwd(x, w, y=None, stream=None):
    """y = w·x·sigmoid(x).  x contiguous (any shape); w: one float32 on the device."""
    import torch
    assert x.is_contiguous()
    if y is None:
        y = torch.empty_like(x)
    with _on(x):
        _check(lib.silu_fwd(_ptr(x), _ptr(w), _ptr(y), x.numel(), _dtype_code(x),
                            _stream(stream, x.device)), "silu_fwd")
    return y


def silu_bwd(dy, x, w, dx=None, dw=None, accumulate=False, workspace=None, stream=None):
    """dx = dy·w·(s + x·s·(1 − s)); dw (+)= Σ dy·x·s.  Returns (dx, dw)."""
    import torch
    assert x.is_contiguous() and dy.is_contiguous()
    code = _dtype_code(x)
    n = x.numel()
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(1, dtype=torch.float32, device=x.device)
    need = lib.silu_bwd_workspace_bytes(n, code)
    with _on(x):
        if workspace is None and need not in (0, SIZE_MAX):
            workspace = _scratch(need, x.device, stream)
        wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib.silu_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(dx), ctypes.c_void_p(dw.data_ptr()),
                            int(bool(accumulate)), _ptr(workspace), wbytes, n, code,
                            _stream(stream, x.device)), "silu_bwd")
    return dx, dw


def norm_bwd_workspace_bytes(N: int, D: int, dtype, layer: bool = False) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code_of_dtype(dtype)
    fn = lib.layernorm_bwd_workspace_bytes if layer else lib.rmsnorm_bwd_workspace_bytes
    return fn(N, D, code)


def rmsnorm_fwd(x, w, eps=1e-5, y=None, stream=None):
    """y = x·r·w per row, r = 1/sqrt(mean x² + eps).  x: [N, D] (unit inner
    stride); w: [D] float32; y has x's type."""
    import torch
    N, D = x.shape
    if y is None:
        y = torch.empty((N, D), dtype=x.dtype, device=x.device)
    with _on(x):
        _check(lib.rmsnorm_fwd(_ptr(x), x.stride(0), _ptr(w), float(eps), _ptr(y), y.stride(0), N,
                               D, _dtype_code(x), _stream(stream, x.device)), "rmsnorm_fwd")
    return y


def layernorm_fwd(x, w, b, eps=1e-5, y=None, stream=None):
    """y = (x − μ)·r·w + b per row.  w, b: [D] float32."""
    import torch
    N, D = x.shape
    if y is None:
        y = torch.empty((N, D), dtype=x.dtype, device=x.device)
    with _on(x):
        _check(lib.layernorm_fwd(_ptr(x), x.stride(0), _ptr(w), _ptr(b), float(eps), _ptr(y),
                                 y.stride(0), N, D, _dtype_code(x), _stream(stream, x.device)),
               "layernorm_fwd")
    return y


def _norm_ws(N, D, code, layer, workspace, device, stream):
    fn = lib.layernorm_bwd_workspace_bytes if layer else lib.rmsnorm_bwd_workspace_bytes
    need = fn(N, D, code)
    if workspace is None and need not in (0, SIZE_MAX):
        workspace = _scratch(need, device, stream)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return workspace, wbytes


def rmsnorm_bwd(x, w, dy, eps=1e-5, dx=None, grad_w=None, accumulate=False, workspace=None,
                stream=None):
    """dx = r·(g − x̂·mean(g·x̂)), g = dy·w; grad_w (+)= Σ_rows dy·x̂.  Returns (dx, grad_w)."""
    import torch
    N, D = x.shape
    code = _dtype_code(x)
    if dx is None:
        dx = torch.empty((N, D), dtype=x.dtype, device=x.device)
    if grad_w is None:
        grad_w = torch.empty(D, dtype=torch.float32, device=x.device)
    with _on(x):
        workspace, wbytes = _norm_ws(N, D, code, False, workspace, x.device, stream)
        _check(lib.rmsnorm_bwd(_ptr(x), x.stride(0), _ptr(w), _ptr(dy), dy.stride(0), float(eps),
                               _ptr(dx), dx.stride(0), _ptr(grad_w), int(bool(accumulate)),
                               _ptr(workspace), wbytes, N, D, code, _stream(stream, x.device)),
               "rmsnorm_bwd")
    return dx, grad_w


def layernorm_bwd(x, w, dy, eps=1e-5, dx=None, grad_w=None, grad_b=None, accumulate=False,
                  workspace=None, stream=None):
    """dx = r·(g − mean g − x̂·mean(g·x̂)); grad_w (+)= Σ dy·x̂; grad_b (+)= Σ dy.
    Returns (dx, grad_w, grad_b)."""
    import torch
    N, D = x.shape
    code = _dtype_code(x)
    if dx is None:
        dx = torch.empty((N, D), dtype=x.dtype, device=x.device)
    if grad_w is None:
        grad_w = torch.empty(D, dtype=torch.float32, device=x.device)
    if grad_b is None:
        grad_b = torch.empty(D, dtype=torch.float32, device=x.device)
    with _on(x):
        workspace, wbytes = _norm_ws(N, D, code, True, workspace, x.device, stream)
        _check(lib.layernorm_bwd(_ptr(x), x.stride(0), _ptr(w), _ptr(dy), dy.stride(0),
                                 float(eps), _ptr(dx), dx.stride(0), _ptr(grad_w), _ptr(grad_b),
                                 int(bool(accumulate)), _ptr(workspace), wbytes, N, D, code,
                                 _stream(stream, x.device)), "layernorm_bwd")
    return dx, grad_w, grad_b


def cluster_wait_timeouts(reset: bool = False) -> int:
    """Waits of the cluster paths' partial-sum exchanges that ran out on the
    current device (zero in correct operation); synchronises the device."""
    n = ctypes.c_uint(0)
    _check(lib.wsf_cluster_wait_timeouts(ctypes.byref(n), int(bool(reset))),
           "wsf_cluster_wait_timeouts")
    return int(n.value)


def selftest_exchange_timeout(count: torch.Tensor, limit_ms: int = 20, stream=None) -> None:
    """Run the cluster exchange's bounded wait where nothing completes it:
    adds selftest_waiting_warps() to the device int32/uint32 scalar `count`
    once the stream reaches it (each waiting warp gives up after limit_ms)."""
    if count.numel() != 1 or count.element_size() != 4 or not count.is_cuda:
        raise TypeError("count must be a one-element 4-byte CUDA tensor")
    with _on(count):
        _check(lib.wsf_selftest_exchange_timeout(_ptr(count), int(limit_ms),
                                                 _stream(stream, count.device)),
               "wsf_selftest_exchange_timeout")


def selftest_waiting_warps() -> int:
    return int(lib.wsf_selftest_waiting_warps())


__all__ = ["lib", "LIB_PATH", "WsfError", "status_string", "cluster_wait_timeouts",
           "selftest_exchange_timeout", "selftest_waiting_warps", "ws_fwd", "ws_bwd", "ws_bwd_noalloc",
           "ws_bwd_atomic", "silu_bwd_atomic", "softmax_fwd", "softmax_bwd", "silu_fwd",
           "silu_bwd", "rmsnorm_fwd", "rmsnorm_bwd", "layernorm_fwd", "layernorm_bwd",
           "ws_bwd_workspace_bytes", "silu_bwd_workspace_bytes", "norm_bwd_workspace_bytes", "F32",
           "F16", "BF16"]
