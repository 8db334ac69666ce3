"""Checks of the seeded input generator (not of the method)."""
import numpy as np
import torch

from inputgen import NORMAL, UNIFORM


def test_splitmix64_published_vector(ig):
    # First three outputs of SplitMix64 from state 0, as published with the
    # reference implementation (Vigna, splitmix64.c).
    assert ig.splitmix64(0, 0) == 0xE220A8397B1DCDAF
    assert ig.splitmix64(0, 1) == 0x6E789E6AA1B965F4
    assert ig.splitmix64(0, 2) == 0x06C45D188009454F


def test_counter_based_subranges(ig):
    full = ig.make((1000,), "f32", NORMAL, 0.0, 1.0, seed=0, stream=0)
    part = ig.make((301,), "f32", NORMAL, 0.0, 1.0, seed=0, stream=0, first=333)
    assert torch.equal(full[333:634], part)
    rows = torch.zeros((7, 13), dtype=torch.float16)
    ig.fill_rows_(rows[:, :10], "f16", 10, UNIFORM, -1, 1, 0, 5, first_row=3)
    ref = ig.make((10, 10), "f16", UNIFORM, -1, 1, 0, 5)
    assert torch.equal(rows[:, :10], ref[3:10]) and torch.count_nonzero(rows[:, 10:]) == 0


def test_streams_and_seeds_differ(ig):
    a = ig.make((64,), "f32", NORMAL, 0, 1, 0, 0)
    b = ig.make((64,), "f32", NORMAL, 0, 1, 0, 1)
    c = ig.make((64,), "f32", NORMAL, 0, 1, 1, 0)
    assert not torch.equal(a, b) and not torch.equal(a, c)


def test_moments(ig):
    n = 1 << 20
    x = ig.make((n,), "f32", NORMAL, 0.0, 2.0, 0, 0).double().numpy()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 2.0) < 0.01
    assert abs((x ** 4).mean() / x.var() ** 2 - 3.0) < 0.05  # normal kurtosis
    u = ig.make((n,), "f16", UNIFORM, -1.0, 1.0, 0, 0).double().numpy()
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.005
    assert abs(u.var() - 1.0 / 3.0) < 0.005


def test_rounded_to_storage_type(ig):
    """The stored value is the nearest storage value to the fp64 draw."""
    x64 = ig.make((4096,), "f32", NORMAL, 0, 1, 0, 9)  # f32 draws (single rounding)
    xb = ig.make((4096,), "bf16", NORMAL, 0, 1, 0, 9)
    assert torch.equal(x64.to(torch.bfloat16), xb) or \
        (x64.to(torch.bfloat16) != xb).sum() <= 2  # double rounding may differ rarely
