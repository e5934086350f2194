"""Pins for the oracle's block-wise quantize / dequantize (section 二 / 逐块量化
and 动态量化 of "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION")."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.blockwise import num_blocks

B = oracle.BLOCK


def codes_at_unit_scale(xn, signed):
    """Codes for normalised values: every block gets a leading 1.0, so its
    absmax is exactly 1 and x / absmax == x."""
    xn = np.asarray(xn, np.float32)
    per = B - 1
    nb = (xn.size + per - 1) // per
    pad = np.zeros(nb * per, np.float32)
    pad[: xn.size] = xn
    rows = np.concatenate([np.ones((nb, 1), np.float32), pad.reshape(nb, per)], axis=1)
    codes, absmax = oracle.quantize_blockwise(rows.ravel(), signed)
    assert np.all(absmax == 1.0)
    return codes.reshape(nb, B)[:, 1:].ravel()[: xn.size]


def all_f32_between(lo, hi):
    a = int(np.array(lo, np.float32).view(np.uint32))
    b = int(np.array(hi, np.float32).view(np.uint32))
    return np.arange(a, b + 1, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("signed", [True, False])
def test_nearest_code_brute_force_exact(signed):
    """Code minimises the exact distance to the map entry over all 256 codes,
    except for inputs in a gap between an exact midpoint and its binary32
    threshold (R4), which must follow the threshold (R7)."""
    rng = np.random.default_rng(1)
    lo = -1.0 if signed else 0.0
    xs = np.concatenate([
        rng.uniform(lo, 1.0, 1500),
        np.sign(rng.uniform(lo, 1.0, 1500)) * 10.0 ** rng.uniform(-8, 0, 1500),
    ]).astype(np.float32)
    m = oracle.dynamic_map(signed)
    t = oracle.thresholds(signed)
    mf = [Fraction(float(v)) for v in m]
    codes = codes_at_unit_scale(xs, signed)
    for x, c in zip(xs, codes):
        xf = Fraction(float(x))
        d = [abs(xf - v) for v in mf]
        best = min(d)
        cands = [i for i in range(256) if d[i] == best]
        if int(c) in cands:
            continue
        # must be the threshold-rounding gap between c and its nearest neighbour
        assert len(cands) == 1 and abs(cands[0] - int(c)) == 1, (x, c, cands)
        i = int(c) if cands[0] > c else int(c) - 1
        mid = (mf[i] + mf[i + 1]) / 2
        assert min(mid, Fraction(float(t[i]))) <= xf <= max(mid, Fraction(float(t[i]))), (x, c, cands)


@pytest.mark.parametrize("signed", [True, False])
def test_every_f32_in_top_decade(signed):
    """Binary32 values in [0.1, 1] -- every one in the top binade and around
    the decade edge, a stride elsewhere -- and their negatives for the signed
    map: the code is a nearest entry by distance to both neighbours; ties
    (exactly on a threshold) take the higher code."""
    xs = np.unique(np.concatenate([
        all_f32_between(0.5, 1.0),          # every value of the top binade
        all_f32_between(0.095, 0.105),      # every value around the decade edge
        all_f32_between(0.1, 0.5)[::7],     # a stride through the rest
    ]))
    m = oracle.dynamic_map(signed).astype(np.float64)
    t = oracle.thresholds(signed)
    for sgn in ([1, -1] if signed else [1]):
        x = (sgn * xs).astype(np.float32)
        c = codes_at_unit_scale(x, signed).astype(np.int64)
        xd = x.astype(np.float64)  # differences below are exact in binary64
        d0 = np.abs(xd - m[c])
        dl = np.where(c > 0, np.abs(xd - m[np.maximum(c - 1, 0)]), np.inf)
        dr = np.where(c < 255, np.abs(xd - m[np.minimum(c + 1, 255)]), np.inf)
        # nearest, up to the binary32 rounding of the thresholds
        slack = np.abs(np.spacing(np.float32(1.0))) * 1.0
        assert np.all(d0 <= dl + slack) and np.all(d0 <= dr + slack)
        # and exactly what "count of thresholds <= x" says
        assert np.array_equal(c, np.searchsorted(t, x, side="right"))
        on_thr = np.isin(x, t)
        if on_thr.any():
            ci = c[on_thr]
            assert np.all(t[ci - 1] == x[on_thr])  # higher code on a tie


@pytest.mark.parametrize("signed", [True, False])
def test_map_values_round_trip(signed):
    m = oracle.dynamic_map(signed)
    c = codes_at_unit_scale(m, signed)
    want = np.arange(256)
    if signed:
        want[127] = 128  # -0.0 takes the code of +0.0 (R7)
    assert np.array_equal(c, want)


def test_zero_inputs_take_code_of_plus_zero():
    x = np.array([1.0, 0.0, -0.0, 1e-30, -1e-30], np.float32)
    c, a = oracle.quantize_blockwise(x, True)
    assert a[0] == 1.0 and list(c[1:3]) == [128, 128]
    assert c[3] == 128 and c[4] == 127  # tiny negative -> -0.0 entry
    c, _ = oracle.quantize_blockwise(np.zeros(3000, np.float32), True)
    assert np.all(c == 128)
    c, a = oracle.quantize_blockwise(np.zeros(3000, np.float32), False)
    assert np.all(c == 0) and np.all(a == 0)
    y = oracle.dequantize_blockwise(c, a, False)
    assert np.all(y == 0)


@pytest.mark.parametrize("n", [1, 2, 2047, 2048, 2049, 4095, 4096, 3 * 2048 + 5])
@pytest.mark.parametrize("signed", [True, False])
def test_block_absmax_and_range(n, signed):
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n).astype(np.float32)
    if not signed:
        x = x * x
    c, a = oracle.quantize_blockwise(x, signed)
    assert c.shape == (n,) and a.shape == (num_blocks(n),)
    y = oracle.dequantize_blockwise(c, a, signed)
    for b in range(num_blocks(n)):
        xb = x[b * B:(b + 1) * B]
        assert a[b] == np.max(np.abs(xb))
        k = int(np.argmax(np.abs(xb)))
        # the absmax element dequantizes to exactly +-absmax (map holds +-1.0)
        assert y[b * B + k] == xb[k]
        yb = y[b * B:(b + 1) * B]
        assert np.all(np.abs(yb) <= a[b])


@pytest.mark.parametrize("signed", [True, False])
def test_outlier_only_touches_its_block(signed):
    """Section 二 / 逐块量化: an outlier's influence stays inside its block."""
    rng = np.random.default_rng(7)
    n = 9 * B + 100
    x = rng.standard_normal(n).astype(np.float32)
    if not signed:
        x = np.abs(x)
    c0, a0 = oracle.quantize_blockwise(x, signed)
    for idx in [0, B - 1, 4 * B + 17, n - 1]:
        x1 = x.copy()
        x1[idx] = np.float32(100.0) * a0[idx // B]
        c1, a1 = oracle.quantize_blockwise(x1, signed)
        b = idx // B
        other = np.ones(num_blocks(n), bool)
        other[b] = False
        assert np.array_equal(a0[other], a1[other])
        mask = np.ones(n, bool)
        mask[b * B:(b + 1) * B] = False
        assert np.array_equal(c0[mask], c1[mask])
        assert a1[b] != a0[b]


@pytest.mark.parametrize("signed", [True, False])
def test_round_trip_error_bound(signed):
    """|x - deq(q(x))| <= absmax * (half the larger neighbouring map gap
    + 2^-23) + one ulp of absmax, per element."""
    rng = np.random.default_rng(3)
    n = 20 * B + 333
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 2, n)).astype(np.float32)
    if not signed:
        x = x * x
    c, a = oracle.quantize_blockwise(x, signed)
    y = oracle.dequantize_blockwise(c, a, signed)
    m = oracle.dynamic_map(signed).astype(np.float64)
    gap = np.zeros(256)
    gap[:-1] = np.diff(m)
    gap[1:] = np.maximum(gap[1:], np.diff(m))
    ab = np.repeat(a, B)[:n].astype(np.float64)
    bound = ab * (0.5 * gap[c] + 2.0 ** -23) + np.spacing(ab.astype(np.float32)).astype(np.float64)
    err = np.abs(x.astype(np.float64) - y.astype(np.float64))
    assert np.all(err <= bound)


def test_blockwise_beats_tensorwise_on_outliers():
    """With one large outlier, per-block scaling keeps the other blocks'
    relative error small, unlike one scale for the whole tensor."""
    rng = np.random.default_rng(11)
    n = 16 * B
    x = rng.standard_normal(n).astype(np.float32)
    x[5] = 1e4
    c, a = oracle.quantize_blockwise(x, True)
    y = oracle.dequantize_blockwise(c, a, True)
    rel_bw = np.abs(y[B:] - x[B:]).mean() / np.abs(x[B:]).mean()
    # whole-tensor normalisation: one scale
    t = oracle.thresholds(True)
    m = oracle.dynamic_map(True)
    s = np.max(np.abs(x))
    yt = m[np.searchsorted(t, x / s, side="right")] * s
    rel_tw = np.abs(yt[B:] - x[B:]).mean() / np.abs(x[B:]).mean()
    assert rel_bw < 0.05 < rel_tw


@pytest.mark.parametrize("signed", [True, False])
def test_codes_are_monotone_within_a_block(signed):
    """Nearest-entry codes of an ascending map never decrease when the input
    does: sorting a block's values sorts its codes (a reversed threshold
    table or a sign slip in the comparison would break this)."""
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(B) * 10.0 ** rng.uniform(-6, 0, B)).astype(np.float32)
    if not signed:
        x = np.abs(x)
    x.sort()
    codes, _ = oracle.quantize_blockwise(x, signed)
    assert np.all(np.diff(codes.astype(np.int32)) >= 0)


@pytest.mark.parametrize("signed", [True, False])
@pytest.mark.parametrize("k", [-40, -7, 1, 30])
def test_power_of_two_scaling_leaves_codes_unchanged(signed, k):
    """Scaling a block by 2^k scales every value and the absmax exactly, so
    x / absmax and the codes are unchanged and the absmax scales by 2^k (a
    swapped operand in the division or a wrong absmax would show here)."""
    rng = np.random.default_rng(100 + k)
    x = (rng.standard_normal(3 * B + 77) * 10.0 ** rng.uniform(-4, 0, 3 * B + 77)).astype(np.float32)
    if not signed:
        x = x * x
    c0, a0 = oracle.quantize_blockwise(x, signed)
    xs = (x * np.float32(2.0 ** k)).astype(np.float32)
    assert np.array_equal(xs / np.float32(2.0 ** k), x)  # no value left the normal range
    c1, a1 = oracle.quantize_blockwise(xs, signed)
    assert np.array_equal(c0, c1)
    assert np.array_equal(a1, (a0 * np.float32(2.0 ** k)).astype(np.float32))
