"""Pins for the oracle's storage-type conversions.

The oracle decodes binary16 / bfloat16 exactly and rounds fp64 results to
them with round-to-nearest-even (the reading taken for the unstated store
rounding of the pages' fp16 stores).  These tests pin both directions against
numpy / torch conversions, against brute-force nearest-value search, and
against the input generator's independently written rounding.
"""
import math

import numpy as np
import pytest
import torch


def _all16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_f16_decode_exhaustive(orc):
    bits = _all16()
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero survives
    assert math.copysign(1.0, orc.f16_to_f64(0x8000)) == -1.0


def test_bf16_decode_exhaustive(orc):
    bits = _all16()
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _finite_patterns(exp_mask):
    bits = _all16().astype(np.uint32)
    return bits[(bits & exp_mask) != exp_mask]


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_encode_roundtrip_and_midpoints(orc, fmt):
    """Every finite value encodes to itself; the midpoint between two
    consecutive positive values goes to the one with an even last bit; a
    point just off the midpoint goes to the nearer one."""
    if fmt == "f16":
        dec, enc, expm = orc.f16_to_f64, orc.f64_to_f16, 0x7C00
    else:
        dec, enc, expm = orc.bf16_to_f64, orc.f64_to_bf16, 0x7F80
    for b in _finite_patterns(expm):
        v = dec(int(b))
        if v == 0.0:
            continue
        assert enc(v) == int(b), (fmt, hex(b))
    # positive finite patterns are ordered by value: b and b+1 are neighbours
    pos = [int(b) for b in _finite_patterns(expm) if b < 0x8000]
    for b in pos[:-1]:
        lo, hi = dec(b), dec(b + 1)
        mid = (lo + hi) / 2.0  # exact in double
        even = b if (b & 1) == 0 else b + 1
        assert enc(mid) == even, (fmt, hex(b))
        assert enc(-mid) == even | 0x8000
        span = hi - lo
        assert enc(mid - span / 8) == b
        assert enc(mid + span / 8) == b + 1


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_encode_specials(orc, fmt):
    enc = orc.f64_to_f16 if fmt == "f16" else orc.f64_to_bf16
    inf = 0x7C00 if fmt == "f16" else 0x7F80
    maxb = 0x7BFF if fmt == "f16" else 0x7F7F
    dec = orc.f16_to_f64 if fmt == "f16" else orc.bf16_to_f64
    assert enc(math.inf) == inf and enc(-math.inf) == inf | 0x8000
    assert (enc(math.nan) & inf) == inf and (enc(math.nan) & ~(inf | 0x8000)) != 0
    assert enc(0.0) == 0 and enc(-0.0) == 0x8000
    top = dec(maxb)
    half_ulp = (top - dec(maxb - 1)) / 2
    assert enc(top + half_ulp * 0.999) == maxb
    assert enc(top + half_ulp) == inf  # tie goes to even = overflow
    # below half the smallest subnormal -> zero; at exactly half -> zero (even)
    tiny = dec(1)
    assert enc(tiny / 2) == 0 and enc(tiny * 0.75) == 1 and enc(-tiny * 0.4) == 0x8000


def test_f16_encode_matches_numpy_random(orc, ig):
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                        rng.uniform(-70000, 70000, 2000)])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)  # numpy rounds double -> half directly
    got = np.array([orc.f64_to_f16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, ref)
    other = np.array([ig.round_f16_bits(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, other)


def test_bf16_encode_nearest_random(orc, ig):
    """No library here rounds double -> bfloat16 in one step, so check the
    definition directly: the encoded value is a nearest bfloat16 value, with
    ties to an even last bit; and the generator's rounding agrees."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)
    for a in v:
        b = orc.f64_to_bf16(float(a))
        got = orc.bf16_to_f64(b)
        for nb in (b - 1, b + 1):
            if 0 <= nb < 65536 and (nb & 0x7F80) != 0x7F80 and ((nb ^ b) & 0x8000) == 0:
                alt = orc.bf16_to_f64(nb)
                assert abs(got - a) <= abs(alt - a)
                if abs(got - a) == abs(alt - a):
                    assert (b & 1) == 0
        assert ig.round_bf16_bits(float(a)) == b


def test_bf16_encode_matches_torch_on_fp32_values(orc):
    """For values representable in binary32, torch's float -> bfloat16
    conversion is a single round-to-nearest-even step."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-20, 20, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f64_to_bf16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, ref)
