"""Pins for the oracle's dynamic-tree codebooks (section 二 / 动态量化 of
"8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION")."""

import os
import struct
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dynamic_map_landmarks.txt")


def _f32_bits(x) -> int:
    return int(np.array(x, np.float32).view(np.uint32))


def _nearest_f32_decimal(num: int, den: int) -> int:
    """Bits of the binary32 nearest to num/den, found by bisection over the
    ordered binary32 bit patterns with 60-digit decimals (independent of the
    oracle's Fraction-based rounding)."""
    getcontext().prec = 60
    target = Decimal(abs(num)) / Decimal(den)
    neg = num < 0

    def val(bits):
        return Decimal(struct.unpack("<f", struct.pack("<I", bits))[0])

    lo, hi = 0, 0x7F800000  # +0 .. +inf, ordered as integers
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if val(mid) <= target:
            lo = mid
        else:
            hi = mid
    dl, dh = target - val(lo), val(hi) - target
    bits = lo if (dl < dh or (dl == dh and lo % 2 == 0)) else hi
    return bits | (0x80000000 if neg else 0)


def _landmarks():
    rows = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            kind, pat, val = line.split()[:3]
            rows.append((kind, int(pat, 16), Fraction(val)))
    return rows


@pytest.mark.parametrize("row", _landmarks(), ids=lambda r: f"{r[0]}-{r[1]:#04x}")
def test_bit_pattern_decode_matches_hand_derived(row):
    kind, pat, exact = row
    if kind == "signed":
        val, sign = oracle.decode_signed(pat)
        assert val == exact
        assert sign == (-1 if pat & 0x80 else 1)
    else:
        assert oracle.decode_unsigned(pat) == exact
    # and the binary32 entry of that value in the map
    m = oracle.dynamic_map(kind == "signed")
    if exact == 0:
        want_neg = kind == "signed" and pat & 0x80
        hits = [i for i in range(256) if m[i] == 0 and bool(np.signbit(m[i])) == bool(want_neg)]
        assert len(hits) == 1
    else:
        bits = _nearest_f32_decimal(exact.numerator, exact.denominator)
        assert bits in {_f32_bits(v) for v in m}


@pytest.mark.parametrize("signed", [True, False])
def test_map_size_order_and_range(signed):
    m = oracle.dynamic_map(signed)
    assert m.shape == (256,) and m.dtype == np.float32
    assert m[0] == (-1.0 if signed else 0.0)
    assert m[255] == 1.0
    d = np.diff(m.astype(np.float64))
    if signed:
        # strictly increasing except the -0.0 / +0.0 pair at 127, 128
        assert np.all(d[:127] > 0) and np.all(d[128:] > 0)
        assert m[127] == 0 and np.signbit(m[127])
        assert m[128] == 0 and not np.signbit(m[128])
    else:
        assert np.all(d > 0)
    assert oracle.zero_code(signed) == (128 if signed else 0)


def test_signed_map_is_symmetric():
    m = oracle.dynamic_map(True)
    for i in range(256):
        assert _f32_bits(m[255 - i]) == (_f32_bits(m[i]) ^ 0x80000000)


@pytest.mark.parametrize("signed,width", [(True, 7), (False, 8)])
def test_points_per_decade_follow_field_widths(signed, width):
    """E leading zeros leave k = width - 1 - E fraction bits: 2**k values in
    the decade (10**-(E+1), 10**-E]; smallest magnitude 10**-(width-1)."""
    m = oracle.dynamic_map(signed)
    pos = np.array([v for v in m if v > 0], np.float64)
    assert pos.size == 2 ** width - 1
    for E in range(width):
        k = width - 1 - E
        lo, hi = nearest(10.0 ** -(E + 1)), nearest(10.0 ** -E)
        cnt = np.count_nonzero((pos > lo) & (pos <= hi))
        assert cnt == 2 ** k, (E, cnt)
    assert pos.min() == nearest(10.0 ** -(width - 1))


def nearest(x):
    return float(np.float32(x))


def test_unsigned_variant_has_the_extra_fraction_bit():
    """The sign bit, reused as fraction, halves the grid step in every decade
    and adds one decade at the bottom (section 二 / 动态量化)."""
    ms, mu = oracle.dynamic_map(True), oracle.dynamic_map(False)
    for E in range(7):
        lo, hi = 10.0 ** -(E + 1), 10.0 ** -E
        s = np.sort(ms[(ms > lo * 1.0000001) & (ms <= hi * 1.0000001)].astype(np.float64))
        u = np.sort(mu[(mu > lo * 1.0000001) & (mu <= hi * 1.0000001)].astype(np.float64))
        assert u.size == 2 * s.size
        gs, gu = np.diff(s).max(initial=0), np.diff(u).max(initial=0)
        if s.size > 1:
            assert gu == pytest.approx(gs / 2, rel=1e-5)
    top_s = np.diff(ms[ms >= np.float32(0.1)].astype(np.float64)).max()
    top_u = np.diff(mu[mu >= np.float32(0.1)].astype(np.float64)).max()
    assert top_s == pytest.approx(0.9 / 64, rel=1e-5)
    assert top_u == pytest.approx(0.9 / 128, rel=1e-5)
    assert mu[mu > 0].min() < ms[ms > 0].min() / 5


@pytest.mark.parametrize("signed", [True, False])
def test_thresholds_are_rounded_midpoints(signed):
    m = oracle.dynamic_map(signed)
    t = oracle.thresholds(signed)
    assert t.shape == (255,) and t.dtype == np.float32
    for i in range(255):
        a, b = Fraction(float(m[i])), Fraction(float(m[i + 1]))
        mid = (a + b) / 2
        ti = Fraction(float(t[i]))
        assert a <= ti <= b
        # no binary32 value is closer to the exact midpoint than t[i]
        for nb in (np.nextafter(t[i], np.float32(-2)), np.nextafter(t[i], np.float32(2))):
            assert abs(Fraction(float(nb)) - mid) >= abs(ti - mid)
    if signed:
        assert t[127] == 0.0
        assert np.all(t[254 - np.arange(255)] == -t)


def test_nearest_f32_against_decimal_bisection():
    rng = np.random.default_rng(0)
    for _ in range(300):
        num = int(rng.integers(1, 10 ** 9)) * int(rng.choice([-1, 1]))
        den = int(rng.integers(1, 10 ** 12))
        got = _f32_bits(oracle.nearest_f32(Fraction(num, den)))
        assert got == _nearest_f32_decimal(num, den)
    # an exact tie between two binary32 values goes to the even significand
    one_plus = Fraction(1) + Fraction(1, 2 ** 24)  # halfway between 1 and 1+2^-23
    assert oracle.nearest_f32(one_plus) == np.float32(1.0)
    three_half = Fraction(1) + Fraction(3, 2 ** 24)
    assert _f32_bits(oracle.nearest_f32(three_half)) == 0x3F800002
