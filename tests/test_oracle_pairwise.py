"""Pins for the oracle's pairwise summation (Higham, Accuracy and Stability
of Numerical Algorithms, 2nd ed., §4.2)."""
import math

import numpy as np


def test_integers_exact(orc):
    for n in [0, 1, 7, 8, 9, 1000, 123457]:
        t = np.arange(n, dtype=np.float64) - n // 3
        assert orc.pairwise_sum(t) == math.fsum(t.tolist())


def test_error_bound(orc):
    """|error| <= (ceil(log2 n) + 8) · 2^-53 · Σ|t| against the correctly
    rounded sum (math.fsum)."""
    rng = np.random.default_rng(5)
    for n in [10, 1000, 1 << 16, 1000003]:
        t = rng.standard_normal(n) * np.exp(rng.uniform(-5, 5, n))
        exact = math.fsum(t.tolist())
        bound = (math.ceil(math.log2(n)) + 8) * 2.0 ** -53 * float(np.abs(t).sum())
        assert abs(orc.pairwise_sum(t) - exact) <= bound


def test_order_of_blocks(orc):
    """The split is at n // 2, blocks of at most eight are added left to right:
    with one huge term, cancelling partners inside one block vanish exactly
    while the same partners in separate halves do not."""
    big = 2.0 ** 60
    t = np.array([big, 1.0, -big, 1.0, 0, 0, 0, 0], dtype=np.float64)  # one block
    assert orc.pairwise_sum(t) == 1.0  # ((big + 1) - big) + 1 = 0 + 1
    t9 = np.array([big, 1.0, 1.0, 1.0, -big, 0, 0, 0, 0], dtype=np.float64)  # halves [0,4) and [4,9)
    assert orc.pairwise_sum(t9) == 0.0  # (big+1+1+1) rounds to big; + (-big) = 0
