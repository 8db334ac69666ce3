"""The oracle's results do not depend on its thread count: rows run in
parallel and the long pairwise sums split into tasks at the same points, so
one thread and four threads give the same bits.  Sizes are chosen so that
the OpenMP task recursion is taken (ranges of more than 2^16 terms)."""
import numpy as np
import pytest
import torch

import oracle


def _run_all(seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(20000, 64, generator=g).to(torch.bfloat16)
    w = torch.randn(64, generator=g)
    dy = torch.randn(20000, generator=g).to(torch.bfloat16)
    out = {}
    ye, ya, yo = oracle.ws_fwd(x, w)
    out["ws_fwd"] = (ye, ya, yo.view(torch.int16).numpy())
    r = oracle.ws_bwd(x, w, dy, block_n=3000)
    out["ws_bwd"] = (r["grad_w"], r["grad_w_abs"], r["partial"], r["dx"].view(torch.int16).numpy())
    xs = torch.randn(300001, generator=g).to(torch.float16)
    gs = torch.randn(300001, generator=g).to(torch.float16)
    rs = oracle.silu_bwd(gs, xs, 0.75)
    out["silu_bwd"] = (rs["dw"], rs["dw_abs"], rs["dx_exact"])
    xm = torch.randn(500, 300, generator=g)
    ymo = oracle.softmax_fwd(xm)
    rm = oracle.softmax_bwd(ymo[1], torch.randn(500, 300, generator=g))
    out["softmax"] = (ymo[0], rm["dx_exact"], rm["s"])
    xn = (torch.randn(3000, 64, generator=g) + 2).to(torch.bfloat16)
    gn = torch.randn(3000, 64, generator=g).to(torch.bfloat16)
    wn = torch.randn(64, generator=g)
    for layer in (False, True):
        f = oracle.norm_fwd(xn, wn, wn if layer else None, 1e-5, layer)
        b = oracle.norm_bwd(xn, wn, gn, 1e-5, layer)
        out[f"norm{int(layer)}"] = (f["y_exact"], b["dx_exact"], b["grad_w"], b["grad_w_abs"],
                                    b["grad_b"], b["grad_b_abs"])
    return out


def test_results_independent_of_thread_count():
    old = oracle.set_threads(1)
    try:
        one = _run_all()
        oracle.set_threads(4)
        four = _run_all()
    finally:
        oracle.set_threads(old)
    for k in one:
        for a, b in zip(one[k], four[k]):
            a, b = np.atleast_1d(np.asarray(a)), np.atleast_1d(np.asarray(b))
            assert a.shape == b.shape, k
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), k
