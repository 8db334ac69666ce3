"""Seeded random configurations of every operator against the fp64 oracle:
storage type, rows and row width (including widths that are not a multiple
of a 16-byte chunk, and rows wider than the register paths), row padding,
pointers misaligned by whole elements, block_n tilings and input scale.
Each case is reproducible from its index; outputs sit inside guard bands."""
import numpy as np
import pytest

import test_gpu_norm as NORM
import test_gpu_parity as PAR
import test_gpu_softmax as SMX

pytestmark = pytest.mark.gpu
DTS = ["f32", "f16", "bf16"]
CASES = 24


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def _shape(rng, max_elems, max_d):
    D = int(rng.choice([int(rng.integers(1, 70)), int(rng.integers(1, max_d + 1))]))
    N = int(rng.integers(1, max(2, min(3000, max_elems // D)) + 1))
    return N, D


@pytest.mark.parametrize("case", range(CASES))
def test_ws_fuzz(wsf, case):
    rng = np.random.default_rng(1000 + case)
    dt = DTS[case % 3]
    N, D = _shape(rng, 1_500_000, 9000)
    pad = int(rng.choice([0, 0, 1, 8, 13]))
    mis = int(rng.choice([0, 0, 1, 3]))
    block_n = int(rng.choice([0, 0, 0, 1, 7, 32, 64]))
    x, w, dy = PAR.make_ws(N, D, dt, seed_shift=3 * case)
    y, dx, gw = PAR.run_ws(wsf, x, w, dy, ld_pad=pad, misalign=mis, block_n=block_n,
                           dy_misalign=int(rng.integers(0, 2)))
    PAR.assert_ws_parity(x, w, dy, y, dx, gw)


@pytest.mark.parametrize("case", range(CASES))
def test_silu_fuzz(wsf, case):
    rng = np.random.default_rng(2000 + case)
    dt = DTS[case % 3]
    n = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(1, 3_000_000))]))
    mis = int(rng.choice([0, 0, 1, 3, 5]))
    x, dy, w = PAR.make_silu(n, dt, w=float(rng.choice([0.75, -1.5, 3.0])))
    PAR.assert_silu_parity(x, dy, w, *PAR.run_silu(wsf, x, dy, w, misalign=mis))


@pytest.mark.parametrize("case", range(CASES))
def test_softmax_fuzz(wsf, case):
    rng = np.random.default_rng(3000 + case)
    dt = DTS[case % 3]
    N, D = _shape(rng, 1_000_000, 40000)
    pad = int(rng.choice([0, 0, 3, 8]))
    mis = int(rng.choice([0, 0, 1]))
    x, dy = SMX._inputs(N, D, dt, seed=case)
    import oracle
    _, yin = oracle.softmax_fwd(x)
    y, dx = SMX._run(wsf, x, dy, yin, pad=pad, mis=mis)
    SMX._check(x, dy, y, dx, yin)


@pytest.mark.parametrize("case", range(CASES))
def test_norm_fuzz(wsf, case):
    rng = np.random.default_rng(4000 + case)
    dt = DTS[case % 3]
    layer = bool(case % 2)
    N, D = _shape(rng, 1_000_000, 12000)
    pad = int(rng.choice([0, 0, 3, 8]))
    mis = int(rng.choice([0, 0, 1]))
    mean = float(rng.choice([0.0, 0.0, 3.0, -40.0]))
    x, w, dy, b = NORM._inputs(N, D, dt, seed=case, mean=mean)
    NORM._check(layer, x, w, dy, b, *NORM._run(wsf, layer, x, w, dy, b, pad=pad, mis=mis))
