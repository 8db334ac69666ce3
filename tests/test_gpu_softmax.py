"""GPU parity of the softmax forward and backward against the fp64 oracle:
register rows of every width class, cluster rows (clusters of 3 to 16 CTAs,
both CTA widths, ragged last slices, more rows than resident clusters), the
element-wise wide/unaligned path, masked (−inf) logits, row strides, guard
bands, windowed rows (odd widths and shifted pointers read as the 16-byte
chunks that cover each row, edges masked), two-pass cluster rows (wider than
32,768 chunks), arrays at mixed offsets, bit
reproducibility, and sampled rows at the measurement size."""
import numpy as np
import pytest
import torch

import oracle
from inputgen import NORMAL
from tolerance import check_elementwise

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTS = ["f32", "f16", "bf16"]


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def _inputs(N, D, dt, seed=0):
    import inputgen
    x = inputgen.make((N, D), dt, NORMAL, 0.0, 2.0, seed, 0)
    dy = inputgen.make((N, D), dt, NORMAL, 0.0, 1.0, seed, 2)
    return x, dy


def _run(wsf, x, dy_host, y_in, pad=0, mis=0):
    """Run forward on x and backward on (y_in, dy) with row stride D + pad and
    pointers shifted by `mis` elements; outputs surrounded by guard bytes."""
    N, D = x.shape
    ld = D + pad

    def place(t):
        b = torch.zeros(N * ld + mis + 16, dtype=t.dtype, device=DEV)
        v = b[mis:mis + N * ld].view(N, ld)[:, :D]
        v.copy_(t.to(DEV))
        return v

    def out():
        b = torch.full((N * ld + mis + 64,), 7.0, dtype=x.dtype, device=DEV)
        return b, b[mis:mis + N * ld].view(N, ld)[:, :D]

    xd, yd, gd = place(x), place(y_in), place(dy_host)
    yb, y = out()
    dxb, dx = out()
    wsf.softmax_fwd(xd, y=y)
    wsf.softmax_bwd(yd, gd, dx=dx)
    torch.cuda.synchronize()
    for b in (yb, dxb):  # the guard bands and row padding keep their fill
        mask = torch.ones_like(b, dtype=torch.bool)
        mask[mis:mis + N * ld].view(N, ld)[:, :D] = False
        assert bool((b[mask] == 7.0).all())
    return y.cpu(), dx.cpu()


def _check(x, dy, y, dx, yin):
    ye, yo = oracle.softmax_fwd(x)
    res = check_elementwise(y, yo, ye)
    assert res and res.clause2 == 0, ("y", res)
    r = oracle.softmax_bwd(yin, dy)
    res = check_elementwise(dx, r["dx"], r["dx_exact"], scale=r["dx_scale"])
    assert res, ("dx", res)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(1, 1), (7, 5), (33, 64), (100, 1000), (9, 2048), (5, 4096),
                                 (3, 8192), (2, 16400), (4, 40000), (1000, 16)])
def test_softmax_parity(wsf, dt, N, D):
    x, dy = _inputs(N, D, dt)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("pad,mis", [(8, 0), (3, 0), (0, 1)])
def test_softmax_strides_alignment(wsf, dt, pad, mis):
    x, dy = _inputs(37, 1024, dt)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin, pad=pad, mis=mis)
    _check(x, dy, y, dx, yin)


def test_softmax_large_logits_and_reproducible(wsf):
    x = torch.tensor([[80.0, 0.0, -80.0, 3.0] * 16], dtype=torch.float32).repeat(5, 1)
    dy = torch.randn(5, 64)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)
    xd, yd, gd = x.to(DEV), yin.to(DEV), dy.to(DEV)
    outs = [(wsf.softmax_fwd(xd), wsf.softmax_bwd(yd, gd)) for _ in range(3)]
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1])


# Cluster rows: 16-byte chunks (8 16-bit or 4 fp32 elements) split over CTAs
# of 1024 chunks (256 threads) for rows of up to 16,384 chunks, else 2048
# chunks (512 threads).
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [
    (700, 16392),   # 16-bit: 2049 chunks, 3 CTAs, the last holding one chunk; more rows than clusters
    (50, 65536),    # 16-bit: 8 CTAs of 256; fp32: 16 CTAs of 256
    (20, 131072),   # 16-bit: 16 CTAs of 256; fp32: 16 CTAs of 512
    (9, 262144),    # 16-bit: 16 CTAs of 512; fp32: beyond the cluster rows (two-pass path)
    (31, 100008),   # ragged last slice
    (13, 50264),
    (3, 50257),     # width not a whole number of chunks (element-wise path)
])
def test_softmax_cluster_rows(wsf, dt, N, D):
    x, dy = _inputs(N, D, dt, seed=N)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)


@pytest.mark.parametrize("dt", DTS)
def test_softmax_cluster_extremes_and_reproducible(wsf, dt):
    # the row maximum in the last CTA's slice, large spreads, a row of equal
    # values, and bit-identical repeats
    N, D = 6, 70000
    x, dy = _inputs(N, D, dt, seed=7)
    x[0, -1] = 60.0
    x[1, 5] = 60.0
    x[2, ::3] = -60.0
    x[3] = 1.5
    x[4, 40000:] = -1e4 if dt != "f16" else -6e4
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)
    xd, yd, gd = x.to(DEV), yin.to(DEV), dy.to(DEV)
    outs = [(wsf.softmax_fwd(xd), wsf.softmax_bwd(yd, gd)) for _ in range(3)]
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1])


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D", [(6, 1000), (6, 40000), (4, 50257), (3, 262144)])
def test_softmax_masked_logits(wsf, dt, N, D):
    # −inf logits (an attention mask): row i keeps columns [0, t_i) and masks
    # the rest, from most of the row down to a single column; the masked
    # spans cover whole warps and whole CTAs of the cluster rows
    x, dy = _inputs(N, D, dt, seed=21)
    keep = [D, D // 2, D // 7, 33, 1, D - 1][:N]
    for i, t in enumerate(keep):
        x[i, t:] = float("-inf")
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)
    for i, t in enumerate(keep):
        assert bool((y[i, t:] == 0).all()) and bool((dx[i, t:] == 0).all())


# Windowed rows: rows that do not start on 16 bytes or whose width is not a
# whole number of chunks, with every array at the same offset (contiguous
# tensors of an odd width, or one shift shared by all); the chunks start at
# each row's first element rounded down to 16 bytes and the edges are masked.
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D,pad,mis", [
    (300, 1001, 0, 0),     # register rows, the offset changes from row to row
    (64, 4097, 0, 0),
    (37, 5, 0, 1),         # tiny rows, every row shifted by one element
    (40, 1024, 3, 1),
    (33, 4096, 0, 1),      # one chunk past a power of two: one more chunk a thread
    (21, 2048, 0, 1),
    (30, 512, 0, 1),
    (50, 50257, 0, 0),     # a GPT-2-sized vocabulary: cluster rows
    (9, 100003, 5, 1),
    (3, 262150, 0, 0),     # wider than the cluster rows (two-pass path)
])
def test_softmax_windowed_rows(wsf, dt, N, D, pad, mis):
    x, dy = _inputs(N, D, dt, seed=D % 89)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin, pad=pad, mis=mis)
    _check(x, dy, y, dx, yin)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("D", [1000, 40000])
def test_softmax_mixed_offsets(wsf, dt, D):
    # arrays at different offsets within their 16-byte blocks take the
    # element-wise path
    N = 20
    x, dy = _inputs(N, D, dt, seed=5)
    _, yin = oracle.softmax_fwd(x)

    def at(t, shift):
        b = torch.zeros(N * D + 16, dtype=t.dtype, device=DEV)
        v = b[shift:shift + N * D].view(N, D)
        v.copy_(t.to(DEV))
        return v

    yb = torch.full((N * D + 16,), 7.0, dtype=x.dtype, device=DEV)
    y = yb[2:2 + N * D].view(N, D)
    dxb = torch.full((N * D + 16,), 7.0, dtype=x.dtype, device=DEV)
    dxv = dxb[3:3 + N * D].view(N, D)
    wsf.softmax_fwd(at(x, 1), y=y)
    wsf.softmax_bwd(at(yin, 0), at(dy, 1), dx=dxv)
    torch.cuda.synchronize()
    assert bool((yb[:2] == 7).all()) and bool((yb[2 + N * D:] == 7).all())
    assert bool((dxb[:3] == 7).all()) and bool((dxb[3 + N * D:] == 7).all())
    _check(x, dy, y.cpu(), dxv.cpu(), yin)


# Two-pass cluster rows: wider than 32,768 chunks; every CTA of a 16-CTA
# cluster streams its slice twice (the second time from L2).
@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N,D,pad,mis", [
    (5, 300000, 0, 0),
    (4, 300007, 0, 0),     # windowed: the offset changes from row to row
    (3, 524288, 8, 1),     # 16-bit: 65,536 chunks; every row shifted by one element
    (100, 140000, 0, 0),   # fp32: 35,000 chunks; more rows than resident clusters
])
def test_softmax_two_pass_rows(wsf, dt, N, D, pad, mis):
    x, dy = _inputs(N, D, dt, seed=D % 83)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin, pad=pad, mis=mis)
    _check(x, dy, y, dx, yin)


@pytest.mark.parametrize("N,D", [(160, 262144), (40, 1048576)])
def test_softmax_two_pass_f32_cluster_sizes(wsf, N, D):
    # binary32 rows take clusters of 8 (160 rows of 1 MB: too many rows in
    # flight for L2 with clusters of 4) and of 16 (rows of 4 MB)
    x, dy = _inputs(N, D, "f32", seed=N)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)


def test_softmax_two_pass_extremes(wsf):
    # the row maximum in the first and in the last slice, a growing maximum
    # within one thread's chunks, masked spans covering whole slices
    N, D = 5, 200000
    x, dy = _inputs(N, D, "f32", seed=9)
    x[0, 0] = 50.0
    x[1, -1] = 50.0
    x[2] = torch.linspace(-30.0, 30.0, D)
    x[3, 1000:] = float("-inf")
    x[4, :150000] = float("-inf")
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)
    assert bool((y[3, 1000:] == 0).all()) and bool((y[4, :150000] == 0).all())


@pytest.mark.parametrize("k", [2, 5, 11, 50])
def test_softmax_two_pass_few_terms(wsf, k):
    """Two-pass binary32 rows whose sum is made of a few terms spread over
    [−4, 0] (the rest masked, or far below): the first pass's sum comes
    from a shorter exponential than the outputs', and with few terms its
    per-term errors do not average out.  Every y within 1e-6 of the exact
    value."""
    N, D = 6, 200000
    g = torch.Generator().manual_seed(k)
    x = torch.full((N, D), float("-inf"))
    x[3:] = -100.0 * torch.rand(N - 3, D, generator=g)
    for r in range(N):
        idx = torch.randperm(D, generator=g)[:k]
        x[r, idx] = -4.0 * torch.rand(k, generator=g)
        x[r, idx[0]] = 0.0
    dy = torch.randn(N, D, generator=g)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin)
    _check(x, dy, y, dx, yin)


@pytest.mark.parametrize("N,D,mis", [(64, 64, 0), (16, 1001, 0), (8, 40000, 0), (4, 300000, 0),
                                     (4, 300007, 1)])
def test_softmax_f32_exponential_range(wsf, N, D, mis):
    """The binary32 exponential (TwoSum-split difference, double-float
    product with log2 e, hardware 2^x, first-order correction) over its
    whole range, on the row, windowed, cluster and two-pass paths: each row
    holds a 0 (its maximum) and logits spread evenly over [−110, 0], so that
    y runs from normal values through subnormal ones to underflow.  Every y
    within 1e-6 of the exact value (or of the binary32 subnormal quantum)."""
    j = np.arange(D, dtype=np.float64)
    frac = (j * 0.6180339887498949 + np.arange(N)[:, None] * 0.137) % 1.0
    x = torch.from_numpy((-110.0 * frac).astype(np.float32))
    x[:, 0] = 0.0
    dy = torch.randn(N, D, generator=torch.Generator().manual_seed(D))
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin, mis=mis)
    _check(x, dy, y, dx, yin)
    ye, _ = oracle.softmax_fwd(x)
    normal = np.abs(ye) >= 2.0 ** -126
    rel = np.abs(y.double().numpy() - ye)[normal] / np.abs(ye)[normal]
    print(f"N={N} D={D}: max relative error of normal y {rel.max():.3g}, "
          f"{int((~normal & (ye > 0)).sum())} subnormal")
    assert rel.max() <= 1e-6


def test_softmax_cluster_no_wait_timeouts(wsf):
    # every cluster launch so far exchanged its partial sums without a wait
    # running out (the counter is per process and device)
    x, dy = _inputs(16, 50000, "bf16", seed=3)
    _, yin = oracle.softmax_fwd(x)
    _run(wsf, x, dy, yin)
    assert wsf.cluster_wait_timeouts() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_softmax_cluster_strides(wsf, dt):
    x, dy = _inputs(40, 40000, dt, seed=2)
    _, yin = oracle.softmax_fwd(x)
    y, dx = _run(wsf, x, dy, yin, pad=8)
    _check(x, dy, y, dx, yin)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["s1", "s2", "s3", "s4"])
def test_softmax_measurement_size_sampled(wsf, name):
    import inputgen
    from inputgen.workloads import WORKLOADS
    wl = WORKLOADS[name]
    x = inputgen.make((wl.N, wl.D), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0, pin=True)
    dy = inputgen.make((wl.N, wl.D), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2, pin=True)
    xd, gd = x.to(DEV), dy.to(DEV)
    y = wsf.softmax_fwd(xd)
    dx = wsf.softmax_bwd(y, gd)
    torch.cuda.synchronize()
    rows = torch.from_numpy(np.unique(np.concatenate([[0, wl.N - 1],
                                                      np.random.default_rng(0).choice(wl.N, 254)])))
    xs, gs = x[rows].contiguous(), dy[rows].contiguous()
    ys = y[rows.to(DEV)].cpu()
    _check(xs, gs, ys, dx[rows.to(DEV)].cpu(), ys)
