"""Dynamic-tree codebooks (oracle).  TEST INFRASTRUCTURE ONLY.

Follows "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (wiki.neutronadmin.com
/news/16836), section 二 / 动态量化: an 8-bit dynamic tree number is made of
  (1) a sign bit,
  (2) an exponent written as the count of leading zero bits,
  (3) an indicator bit (the first 1) saying that the rest is a linear value,
  (4) the linear fraction in the remaining bits.
The optimizer variant ("dynamic quantization") drops the sign for the always
positive second moment and spends that bit on the fraction.

The page fixes the four fields but not the numbers.  Readings taken here:
  R1  the zero-run exponent is decimal: E leading zeros scale by 10**-E (the
      page says the type keeps more *decimal* places);
  R2  the k fraction bits j pick the right end points of a linear grid on
      (0.1, 1]:  |value| = 10**-E * (0.1 + 0.9 * (j + 1) / 2**k).  So 1.0 is
      exact, each decade (10**-(E+1), 10**-E] holds 2**k points and adjacent
      decades tile without a gap or a duplicate;
  R2' the pattern with no indicator bit (all tail bits zero) is zero; in the
      signed type it carries its sign, giving -0.0 and +0.0;
  R3  a stored code is the index of its value in the ascending map (with -0.0
      before +0.0), not the bit pattern;
  R4  threshold i is the binary32 value nearest to the exact midpoint of map
      entries i and i+1 (both already binary32), ties to even.

Parity: pinned by tests/test_oracle_codebook.py (field counts per decade,
monotonicity, symmetry, extreme values, the unsigned variant's finer grid,
bit-pattern decode against values derived by hand in tests/golden/).
"""

from __future__ import annotations

from fractions import Fraction
from functools import lru_cache

import numpy as np

#: Block length of the block-wise normalisation (section 二 / 逐块量化).
BLOCK = 2048


def nearest_f32(q: Fraction) -> np.float32:
    """Binary32 value nearest to the exact rational ``q`` (ties to even).

    ``float(q)`` is the correctly rounded binary64 value; rounding that once
    more to binary32 can be off by one unit (double rounding), so the three
    binary32 candidates around it are compared in exact arithmetic.
    """
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = -q if q < 0 else q
    f = np.float32(float(a))
    cands = [
        np.nextafter(f, np.float32(0.0)),
        f,
        np.nextafter(f, np.float32(np.inf)),
    ]
    best = None
    best_d = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - a)
        if best is None or d < best_d:
            best, best_d = c, d
        elif d == best_d:
            # tie: keep the candidate whose significand is even
            if int(np.array(c, np.float32).view(np.uint32)) & 1 == 0:
                best = c
    return np.float32(sign * best)


def _magnitude(E: int, k: int, j: int) -> Fraction:
    """R1 + R2: 10**-E * (0.1 + 0.9 * (j + 1) / 2**k), exactly."""
    return Fraction(1, 10 ** E) * (Fraction(1, 10) + Fraction(9, 10) * Fraction(j + 1, 2 ** k))


def _decode_tail(bits: int, width: int):
    """Decode the sign-less tail of ``width`` bits.

    Returns ``None`` for the all-zero tail (no indicator bit: zero), otherwise
    the exact magnitude.  E = number of leading zeros, then the indicator 1,
    then k = width - 1 - E fraction bits holding j.
    """
    if bits == 0:
        return None
    E = 0
    for pos in range(width - 1, -1, -1):
        if (bits >> pos) & 1:
            break
        E += 1
    k = width - 1 - E
    j = bits & ((1 << k) - 1)
    return _magnitude(E, k, j)


def decode_signed(pattern: int):
    """Exact value of a signed 8-bit dynamic tree pattern.

    Bit 7 is the sign; bits 6..0 are the tail.  Returns ``(Fraction, sign)``
    where sign is -1 or +1 (kept separately so that -0 and +0 stay distinct).
    """
    if not 0 <= pattern < 256:
        raise ValueError("pattern out of range")
    sign = -1 if pattern & 0x80 else 1
    mag = _decode_tail(pattern & 0x7F, 7)
    if mag is None:
        return Fraction(0), sign
    return sign * mag, sign


def decode_unsigned(pattern: int) -> Fraction:
    """Exact value of an unsigned 8-bit pattern: all 8 bits form the tail."""
    if not 0 <= pattern < 256:
        raise ValueError("pattern out of range")
    mag = _decode_tail(pattern, 8)
    return Fraction(0) if mag is None else mag


@lru_cache(maxsize=None)
def _map_exact(signed: bool):
    """The 256 exact values in ascending order (R3), as (Fraction, sign)."""
    if signed:
        vals = [decode_signed(p) for p in range(256)]
    else:
        vals = [(decode_unsigned(p), 1) for p in range(256)]
    # ascending by value; the zero pair is ordered -0.0 then +0.0
    vals.sort(key=lambda vs: (vs[0], vs[1]))
    return tuple(vals)


@lru_cache(maxsize=None)
def _map_f32(signed: bool) -> bytes:
    out = np.empty(256, np.float32)
    for i, (v, s) in enumerate(_map_exact(signed)):
        if v == 0:
            out[i] = np.float32(-0.0) if s < 0 else np.float32(0.0)
        else:
            out[i] = nearest_f32(v)
    return out.tobytes()


def dynamic_map(signed: bool) -> np.ndarray:
    """The 256-entry binary32 codebook, ascending; index = stored code."""
    return np.frombuffer(_map_f32(bool(signed)), np.float32).copy()


@lru_cache(maxsize=None)
def _thr_f32(signed: bool) -> bytes:
    m = dynamic_map(signed)
    t = np.empty(255, np.float32)
    for i in range(255):
        mid = (Fraction(float(m[i])) + Fraction(float(m[i + 1]))) / 2
        t[i] = nearest_f32(mid)
    return t.tobytes()


def thresholds(signed: bool) -> np.ndarray:
    """R4: the 255 decision thresholds between neighbouring codes."""
    return np.frombuffer(_thr_f32(bool(signed)), np.float32).copy()


def zero_code(signed: bool) -> int:
    """Code of +0.0: 128 in the signed map, 0 in the unsigned map."""
    m = dynamic_map(signed)
    for i in range(256):
        if m[i] == 0 and not np.signbit(m[i]):
            return i
    raise AssertionError("map has no +0.0")
