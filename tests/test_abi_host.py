"""Host-only checks of the C ABI: the library loads, exports every entry
point that include/wsf.h declares, answers its workspace queries, and
rejects bad arguments before touching any device (no GPU needed: every
pointer here is a fake address that must never be dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__._cuda_build_module().build()
    import backward_ws_fwd_gb300 as m
    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "wsf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(wsf):
    names = _declared_functions()
    assert {"ws_fwd", "ws_bwd", "silu_fwd", "silu_bwd", "ws_bwd_workspace_bytes",
            "silu_bwd_workspace_bytes", "wsf_status_string", "wsf_version"} <= set(names)
    for n in names:
        assert hasattr(wsf.lib, n), n


def test_selftest_exchange_timeout_rejects(wsf):
    f = wsf.lib.wsf_selftest_exchange_timeout
    assert f(None, 20, None) == -1
    assert f(ctypes.c_void_p(0x1002), 20, None) == -7  # not 4-byte aligned
    assert f(ctypes.c_void_p(0x1000), 0, None) == -8
    assert f(ctypes.c_void_p(0x1000), 1001, None) == -8
    assert wsf.selftest_waiting_warps() == 4


def test_cluster_wait_timeouts_rejects(wsf):
    n = ctypes.c_uint(7)
    assert wsf.lib.wsf_cluster_wait_timeouts(None, 0) == -1
    assert wsf.lib.wsf_cluster_wait_timeouts(ctypes.byref(n), 2) == -8
    assert n.value == 7


def test_status_strings(wsf):
    for code in range(-9, 1):
        s = wsf.status_string(code)
        assert s and s != "unknown status"
    assert wsf.status_string(-100) == "unknown status"


def _plane_bytes(P, D):
    """One binary32 plane of P·D partial sums, rounded up to 256 bytes."""
    return (P * D + 63) // 64 * 64 * 4


def test_workspace_queries(wsf):
    q = wsf.lib.ws_bwd_workspace_bytes
    # the worked shape: 100 rows in 32-row tiles -> 4 partial rows of 64,
    # held as compensated pairs (a plane of high parts, one of low parts)
    assert q(100, 64, wsf.F32, 32) == 2 * 4 * 64 * 4
    assert q(100, 64, wsf.F32, 1) == 2 * _plane_bytes(100, 64)
    assert q(0, 64, wsf.F32, 0) == 0 and q(5, 0, wsf.F16, 0) == 0
    assert q(-1, 4, wsf.F32, 0) == wsf.SIZE_MAX
    assert q(4, 4, 7, 0) == wsf.SIZE_MAX and q(4, 4, wsf.F32, -1) == wsf.SIZE_MAX
    for N, D, dt in [(1 << 20, 1024, wsf.BF16), (1 << 24, 64, wsf.F16), (4096, 65536, wsf.F32),
                     (7, 5, wsf.F32), (1, 1, wsf.F16)]:
        # at most 912 CTAs per launch (tiles x 256-chunk column slices), at
        # most one tile per 64 rows, at least one
        es = 4 if dt == wsf.F32 else 2
        slices = -(-(-(-(D * es) // 16)) // 256)
        P = max(1, min(-(-N // 64), 912 // slices))
        assert q(N, D, dt, 0) == 2 * _plane_bytes(P, D), (N, D, dt)
    # the measurement workloads fit the no-allocation entry point's scratch
    assert max(q(1 << 20, 1024, wsf.BF16, 0), q(1 << 24, 64, wsf.F16, 0),
               q(4096, 65536, wsf.F32, 0)) <= 8 << 20
    s = wsf.lib.silu_bwd_workspace_bytes
    assert s(0, wsf.F16) == 0 and s(1, wsf.F16) == 2 * 256 and s(-1, wsf.F16) == wsf.SIZE_MAX
    assert s(8192 * 4096, wsf.F16) == 2 * _plane_bytes(1216, 1)


F = 0x10000000  # fake, well-aligned device addresses; never dereferenced


def _p(a):
    return ctypes.c_void_p(a)


def test_ws_fwd_rejects(wsf):
    L = wsf.lib
    s = None
    assert L.ws_fwd(_p(F), 64, _p(2 * F), _p(3 * F), 100, 64, 9, s) == wsf.ERR_BAD_DTYPE
    assert L.ws_fwd(_p(F), 64, _p(2 * F), _p(3 * F), -1, 64, 0, s) == wsf.ERR_BAD_SHAPE
    assert L.ws_fwd(_p(F), 64, _p(2 * F), _p(3 * F), 100, -3, 0, s) == wsf.ERR_BAD_SHAPE
    assert L.ws_fwd(_p(F), 63, _p(2 * F), _p(3 * F), 100, 64, 0, s) == wsf.ERR_BAD_STRIDE
    assert L.ws_fwd(None, 64, _p(2 * F), _p(3 * F), 100, 64, 0, s) == wsf.ERR_NULL_PTR
    assert L.ws_fwd(_p(F), 64, None, _p(3 * F), 100, 64, 0, s) == wsf.ERR_NULL_PTR
    assert L.ws_fwd(_p(F), 64, _p(2 * F), None, 100, 64, 0, s) == wsf.ERR_NULL_PTR
    assert L.ws_fwd(_p(F + 1), 64, _p(2 * F), _p(3 * F), 100, 64, 1, s) == wsf.ERR_MISALIGNED
    assert L.ws_fwd(_p(F), 64, _p(2 * F + 2), _p(3 * F), 100, 64, 1, s) == wsf.ERR_MISALIGNED
    # y inside x
    assert L.ws_fwd(_p(F), 64, _p(2 * F), _p(F + 256), 100, 64, 0, s) == wsf.ERR_OVERLAP
    # overflowing sizes
    assert L.ws_fwd(_p(F), 1 << 62, _p(2 * F), _p(3 * F), 4, 64, 0, s) == wsf.ERR_BAD_SHAPE
    # empty: nothing to do, nothing enqueued
    assert L.ws_fwd(None, 0, None, None, 0, 64, 0, s) == wsf.OK


def test_ws_bwd_rejects(wsf):
    L = wsf.lib
    s = None
    need = L.ws_bwd_workspace_bytes(100, 64, 0, 0)
    args = dict(x=F, ldx=64, w=2 * F, dy=3 * F, dx=4 * F, lddx=64, gw=5 * F, acc=0, ws=6 * F,
                wsb=need, bn=0, N=100, D=64, dt=0)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.ws_bwd(_p(a["x"]) if a["x"] else None, a["ldx"], _p(a["w"]) if a["w"] else None,
                        _p(a["dy"]) if a["dy"] else None, _p(a["dx"]) if a["dx"] else None, a["lddx"],
                        _p(a["gw"]) if a["gw"] else None, a["acc"], _p(a["ws"]) if a["ws"] else None,
                        a["wsb"], a["bn"], a["N"], a["D"], a["dt"], s)

    assert call(dt=3) == wsf.ERR_BAD_DTYPE
    assert call(N=-1) == wsf.ERR_BAD_SHAPE
    assert call(bn=-2) == wsf.ERR_BAD_ARG
    assert call(acc=2) == wsf.ERR_BAD_ARG
    assert call(lddx=10) == wsf.ERR_BAD_STRIDE
    assert call(ldx=10) == wsf.ERR_BAD_STRIDE
    for k in ["x", "w", "dy", "dx", "gw"]:
        assert call(**{k: 0}) == wsf.ERR_NULL_PTR, k
    assert call(ws=0) == wsf.ERR_WORKSPACE
    assert call(wsb=need - 1) == wsf.ERR_WORKSPACE
    assert call(bn=32, wsb=need) == wsf.ERR_WORKSPACE or \
        L.ws_bwd_workspace_bytes(100, 64, 0, 32) <= need
    assert call(dx=F + 64) == wsf.ERR_OVERLAP
    assert call(gw=3 * F) == wsf.ERR_OVERLAP
    assert call(ws=4 * F + 128) == wsf.ERR_OVERLAP
    assert call(dx=4 * F + 2) == wsf.ERR_MISALIGNED


def test_ws_bwd_noalloc_rejects(wsf):
    """The no-allocation entry point checks its arguments as ws_bwd does, in
    the same order, before its scratch limit and before touching a device."""
    L = wsf.lib
    N, D = 2048, 1024  # one-row tiles of 1024 fp32 need 16 MiB, over the 8 MiB scratch

    def call(x=F, N=N, bn=0, dt=0, acc=0, ld=D):
        return L.ws_bwd_noalloc(_p(x) if x else None, ld, _p(2 * F), _p(3 * F), _p(4 * F), ld,
                                _p(5 * F), acc, bn, N, D, dt, None)

    assert call(bn=1) == wsf.ERR_WORKSPACE
    assert call(x=0, bn=1) == wsf.ERR_NULL_PTR          # a NULL pointer wins, as from ws_bwd
    assert call(dt=7, bn=1) == wsf.ERR_BAD_DTYPE
    assert call(N=-1) == wsf.ERR_BAD_SHAPE
    assert call(acc=3, bn=1) == wsf.ERR_BAD_ARG
    assert call(ld=D - 1, bn=1) == wsf.ERR_BAD_STRIDE
    assert call(x=4 * F + 64) == wsf.ERR_OVERLAP         # dx over x
    assert call(x=F + 1, dt=1, bn=1) == wsf.ERR_MISALIGNED
    assert L.ws_bwd_noalloc(None, 0, None, None, None, 0, None, 0, 0, 0, 0, 0, None) == wsf.OK


def test_silu_rejects(wsf):
    L = wsf.lib
    s = None
    assert L.silu_fwd(_p(F), _p(2 * F), _p(3 * F), 100, 5, s) == wsf.ERR_BAD_DTYPE
    assert L.silu_fwd(_p(F), _p(2 * F), _p(3 * F), -1, 1, s) == wsf.ERR_BAD_SHAPE
    assert L.silu_fwd(None, _p(2 * F), _p(3 * F), 100, 1, s) == wsf.ERR_NULL_PTR
    assert L.silu_fwd(_p(F), None, _p(3 * F), 100, 1, s) == wsf.ERR_NULL_PTR
    assert L.silu_fwd(_p(F), _p(2 * F), _p(F + 10), 100, 1, s) == wsf.ERR_OVERLAP
    assert L.silu_fwd(_p(F + 1), _p(2 * F), _p(3 * F), 100, 1, s) == wsf.ERR_MISALIGNED
    assert L.silu_fwd(None, None, None, 0, 1, s) == wsf.OK
    need = L.silu_bwd_workspace_bytes(100, 1)
    ok = dict(dy=F, x=2 * F, w=3 * F, dx=4 * F, dw=5 * F, acc=0, ws=6 * F, wsb=need, n=100, dt=1)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        P = lambda v: _p(v) if v else None  # noqa: E731
        return L.silu_bwd(P(a["dy"]), P(a["x"]), P(a["w"]), P(a["dx"]), P(a["dw"]), a["acc"],
                          P(a["ws"]), a["wsb"], a["n"], a["dt"], s)

    assert call(dt=-1) == wsf.ERR_BAD_DTYPE
    assert call(n=-5) == wsf.ERR_BAD_SHAPE
    assert call(acc=3) == wsf.ERR_BAD_ARG
    for k in ["dy", "x", "w", "dx", "dw"]:
        assert call(**{k: 0}) == wsf.ERR_NULL_PTR, k
    assert call(ws=0) == wsf.ERR_WORKSPACE
    assert call(wsb=need - 4) == wsf.ERR_WORKSPACE
    assert call(dx=2 * F + 100) == wsf.ERR_OVERLAP
    assert call(dw=6 * F + 8) == wsf.ERR_OVERLAP
    assert call(x=2 * F + 1) == wsf.ERR_MISALIGNED


def test_atomic_variants_reject(wsf):
    L = wsf.lib
    s = None
    ok = dict(x=F, ldx=64, w=2 * F, dy=3 * F, dx=4 * F, lddx=64, gw=5 * F, acc=0, N=100, D=64, dt=1)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        P = lambda v: _p(v) if v else None  # noqa: E731
        return L.ws_bwd_atomic(P(a["x"]), a["ldx"], P(a["w"]), P(a["dy"]), P(a["dx"]), a["lddx"],
                               P(a["gw"]), a["acc"], a["N"], a["D"], a["dt"], s)

    assert call(dt=4) == wsf.ERR_BAD_DTYPE
    assert call(N=-1) == wsf.ERR_BAD_SHAPE
    assert call(acc=5) == wsf.ERR_BAD_ARG
    assert call(ldx=3) == wsf.ERR_BAD_STRIDE
    assert call(gw=0) == wsf.ERR_NULL_PTR
    assert call(dy=3 * F + 2) == wsf.ERR_MISALIGNED  # staged layout only
    assert call(D=60, ldx=60, lddx=60) == wsf.ERR_MISALIGNED
    assert call(dx=F + 16) == wsf.ERR_OVERLAP
    sa = lambda **kw: L.silu_bwd_atomic(*(  # noqa: E731
        [_p(kw.get("dy", F)), _p(kw.get("x", 2 * F)), _p(kw.get("w", 3 * F)),
         _p(kw.get("dx", 4 * F)) if kw.get("dx", 4 * F) else None,
         _p(kw.get("dw", 5 * F)) if kw.get("dw", 5 * F) else None,
         kw.get("acc", 0), kw.get("n", 100), kw.get("dt", 1), s]))
    assert sa(dt=9) == wsf.ERR_BAD_DTYPE
    assert sa(n=-3) == wsf.ERR_BAD_SHAPE
    assert sa(acc=2) == wsf.ERR_BAD_ARG
    assert sa(dw=0) == wsf.ERR_NULL_PTR
    assert sa(dx=2 * F + 50) == wsf.ERR_OVERLAP


def test_softmax_rejects(wsf):
    L = wsf.lib
    s = None
    assert L.softmax_fwd(_p(F), 64, _p(2 * F), 64, 10, 64, 7, s) == wsf.ERR_BAD_DTYPE
    assert L.softmax_fwd(_p(F), 64, _p(2 * F), 64, -1, 64, 1, s) == wsf.ERR_BAD_SHAPE
    assert L.softmax_fwd(_p(F), 63, _p(2 * F), 64, 10, 64, 1, s) == wsf.ERR_BAD_STRIDE
    assert L.softmax_fwd(None, 64, _p(2 * F), 64, 10, 64, 1, s) == wsf.ERR_NULL_PTR
    assert L.softmax_fwd(_p(F), 64, _p(F + 64), 64, 10, 64, 1, s) == wsf.ERR_OVERLAP
    assert L.softmax_fwd(_p(F + 1), 64, _p(2 * F), 64, 10, 64, 1, s) == wsf.ERR_MISALIGNED
    assert L.softmax_fwd(None, 0, None, 0, 0, 64, 1, s) == wsf.OK
    assert L.softmax_bwd(_p(F), 64, _p(2 * F), 64, _p(3 * F), 64, 10, 64, 9, s) == wsf.ERR_BAD_DTYPE
    assert L.softmax_bwd(_p(F), 64, _p(2 * F), 64, _p(3 * F), 8, 10, 64, 1, s) == wsf.ERR_BAD_STRIDE
    assert L.softmax_bwd(_p(F), 64, None, 64, _p(3 * F), 64, 10, 64, 1, s) == wsf.ERR_NULL_PTR
    assert L.softmax_bwd(_p(F), 64, _p(2 * F), 64, _p(2 * F + 2), 64, 10, 64, 1, s) == \
        wsf.ERR_OVERLAP


def test_norm_workspace_queries(wsf):
    r, l = wsf.lib.rmsnorm_bwd_workspace_bytes, wsf.lib.layernorm_bwd_workspace_bytes
    # 100 rows: ceil(100/64) = 2 row tiles of D fp32 partials (twice for LayerNorm)
    assert r(100, 64, wsf.F32) == 2 * 64 * 4 and l(100, 64, wsf.F32) == 2 * 2 * 64 * 4
    assert r(65536, 4096, wsf.BF16) == 912 * 4096 * 4
    assert l(65536, 4096, wsf.BF16) == 2 * 912 * 4096 * 4
    assert r(0, 64, wsf.F16) == 0 and l(5, 0, wsf.F16) == 0
    assert r(-1, 4, wsf.F32) == wsf.SIZE_MAX and l(4, 4, 3) == wsf.SIZE_MAX
    assert r(1 << 20, 1 << 60, wsf.F32) == wsf.SIZE_MAX  # 16 tiles · 2^60 · 4 bytes overflows


def test_norm_rejects(wsf):
    L = wsf.lib
    s = None
    eps = 1e-5
    rf = lambda x=F, ldx=64, w=2 * F, e=eps, y=3 * F, ldy=64, N=10, D=64, dt=1: L.rmsnorm_fwd(
        _p(x) if x else None, ldx, _p(w) if w else None, e, _p(y) if y else None, ldy, N, D, dt, s)
    assert rf(dt=5) == wsf.ERR_BAD_DTYPE
    assert rf(N=-1) == wsf.ERR_BAD_SHAPE
    assert rf(e=-1.0) == wsf.ERR_BAD_ARG and rf(e=float("nan")) == wsf.ERR_BAD_ARG
    assert rf(e=float("inf")) == wsf.ERR_BAD_ARG
    assert rf(ldx=63) == wsf.ERR_BAD_STRIDE and rf(ldy=8) == wsf.ERR_BAD_STRIDE
    assert rf(x=0) == wsf.ERR_NULL_PTR and rf(w=0) == wsf.ERR_NULL_PTR
    assert rf(x=F + 1) == wsf.ERR_MISALIGNED and rf(w=2 * F + 2) == wsf.ERR_MISALIGNED
    assert rf(y=F + 64) == wsf.ERR_OVERLAP and rf(y=2 * F - 100) == wsf.ERR_OVERLAP
    assert rf(x=0, w=0, y=0, N=0) == wsf.OK and rf(x=0, w=0, y=0, D=0) == wsf.OK
    # LayerNorm needs b; b must not overlap y
    assert L.layernorm_fwd(_p(F), 64, _p(2 * F), None, eps, _p(3 * F), 64, 10, 64, 1, s) == \
        wsf.ERR_NULL_PTR
    assert L.layernorm_fwd(_p(F), 64, _p(2 * F), _p(3 * F + 8), eps, _p(3 * F), 64, 10, 64, 1,
                           s) == wsf.ERR_OVERLAP

    need_r = L.rmsnorm_bwd_workspace_bytes(10, 64, 1)
    need_l = L.layernorm_bwd_workspace_bytes(10, 64, 1)

    def rb(x=F, w=2 * F, dy=3 * F, lddy=64, e=eps, dx=4 * F, lddx=64, gw=5 * F, acc=0, ws=6 * F,
           wsb=need_r, N=10, D=64, dt=1):
        P = lambda a: _p(a) if a else None
        return L.rmsnorm_bwd(P(x), 64, P(w), P(dy), lddy, e, P(dx), lddx, P(gw), acc, P(ws), wsb,
                             N, D, dt, s)

    assert rb(dt=-1) == wsf.ERR_BAD_DTYPE
    assert rb(D=-2) == wsf.ERR_BAD_SHAPE
    assert rb(acc=2) == wsf.ERR_BAD_ARG and rb(e=-0.5) == wsf.ERR_BAD_ARG
    assert rb(lddy=10) == wsf.ERR_BAD_STRIDE and rb(lddx=63) == wsf.ERR_BAD_STRIDE
    assert rb(dy=0) == wsf.ERR_NULL_PTR and rb(gw=0) == wsf.ERR_NULL_PTR
    assert rb(gw=5 * F + 2) == wsf.ERR_MISALIGNED and rb(dx=4 * F + 1) == wsf.ERR_MISALIGNED
    assert rb(ws=0) == wsf.ERR_WORKSPACE and rb(wsb=need_r - 4) == wsf.ERR_WORKSPACE
    assert rb(dx=3 * F + 64) == wsf.ERR_OVERLAP          # dx over dy
    assert rb(gw=4 * F + 256) == wsf.ERR_OVERLAP         # grad_w inside dx
    assert rb(ws=2 * F + 128) == wsf.ERR_OVERLAP         # workspace over w
    assert rb(ws=5 * F - 4) == wsf.ERR_OVERLAP           # workspace over grad_w
    assert rb(x=0, dy=0, dx=0, w=0, ws=0, wsb=0, D=0) == wsf.OK
    assert rb(x=0, dy=0, dx=0, w=0, ws=0, wsb=0, N=0, gw=0) == wsf.ERR_NULL_PTR  # D > 0 needs grad_w

    def lb(gw=5 * F, gb=7 * F, ws=6 * F, wsb=need_l):
        P = lambda a: _p(a) if a else None
        return L.layernorm_bwd(_p(F), 64, _p(2 * F), _p(3 * F), 64, eps, _p(4 * F), 64, P(gw), P(gb),
                               0, P(ws), wsb, 10, 64, 1, s)

    assert lb(gb=0) == wsf.ERR_NULL_PTR
    assert lb(wsb=need_r) == wsf.ERR_WORKSPACE   # LayerNorm needs both partial blocks
    assert lb(gb=5 * F + 128) == wsf.ERR_OVERLAP  # grad_b over grad_w
    assert lb(gb=6 * F + 256) == wsf.ERR_OVERLAP  # grad_b inside the workspace
