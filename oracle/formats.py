"""Exact decoding and round-to-nearest-even for e4m3 (fp8 "e4m3fn") and e2m1 (fp4).

NVFP4 (README "Frontier MoE on consumer Blackwell (SM120)", §"GLM-5.2 (753B)"
¶1: e2m1 values x e4m3 block-16 scale x fp32 per-tensor scale_2) is built from
these two small formats.

Rounding rule used everywhere in this library: a quantity defined as a ratio
a/d of two exactly known numbers is rounded ONCE, to nearest, ties to the even
code, saturating to the largest finite value.  The fp64 path never rounds the
ratio itself: it compares ``2*a`` against ``d * (lo + hi)``, the doubled
midpoint of the two neighbouring representable values, and all those products
are exact in fp64 because every operand has few significant bits (e2m1: 2,
e4m3: 4, midpoints: 5, fp32 factors: 24).  The ``*_fraction`` functions do the
same with Python ``fractions.Fraction`` and serve as an exact cross-check.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

# ---------------------------------------------------------------- e2m1 (fp4)
# code bits: s | e e | m ; exponent bias 1; no inf/NaN.
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAG_FRAC = [Fraction(v).limit_denominator() for v in E2M1_MAG]


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    """fp64 value of 4-bit codes (bit 3 = sign, bits 0..2 = magnitude index)."""
    code = np.asarray(code).astype(np.int64)
    mag = E2M1_MAG[code & 7]
    return np.where(code & 8, -mag, mag)


# ---------------------------------------------------------------- e4m3 (fp8)
def _e4m3_value_frac(code: int):
    """Exact value of an e4m3fn code, or None for NaN (0x7F / 0xFF)."""
    s = code >> 7
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        v = Fraction(m, 8) * Fraction(1, 64)          # subnormal: m/8 * 2^-6
    else:
        v = Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -v if s else v


E4M3_VALUE_FRAC = [_e4m3_value_frac(c) for c in range(256)]
E4M3_VALUE = np.array([np.nan if v is None else float(v) for v in E4M3_VALUE_FRAC])
# non-negative finite codes 0..126 are increasing in value
E4M3_POS = E4M3_VALUE[:127].copy()
E4M3_MAX_CODE = 126          # 448
assert np.all(np.diff(E4M3_POS) > 0)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    return E4M3_VALUE[np.asarray(code).astype(np.int64)]


def _rne_ratio(a, d, pos_values: np.ndarray, even_is_code_parity: bool = True):
    """Index i of RNE(a/d) over increasing ``pos_values`` (saturating).

    a >= 0 and d > 0 are fp64 arrays (broadcastable) holding exact values, and
    d * pos_values[i] must be exact in fp64.  The rounded quotient is never
    formed: the first guess from a/d is corrected by exact comparisons
    against neighbouring values, and the final choice between the two
    neighbours compares 2*a with d*(lo + hi).
    """
    a, d = np.broadcast_arrays(np.asarray(a, np.float64), np.asarray(d, np.float64))
    n = len(pos_values)
    i = np.searchsorted(pos_values, a / d, side="right") - 1
    i = np.clip(i, 0, n - 1)
    for _ in range(3):                       # exact fix-up of the float guess
        down = (i > 0) & (a < d * pos_values[i])
        i = np.where(down, i - 1, i)
        up = (i < n - 1) & (a >= d * pos_values[np.minimum(i + 1, n - 1)])
        i = np.where(up, i + 1, i)
    # now pos[i] <= a/d < pos[i+1] (or i = n-1: saturate)
    top = i >= n - 1
    hi_i = np.minimum(i + 1, n - 1)
    twice_mid_times_d = d * (pos_values[i] + pos_values[hi_i])
    two_a = 2.0 * a
    go_up = two_a > twice_mid_times_d
    tie = two_a == twice_mid_times_d
    # ties go to the even code: codes are the indices themselves
    go_up = go_up | (tie & ((i & 1) == 1))
    return np.where(top, n - 1, np.where(go_up, i + 1, i))


def e4m3_rne_ratio(a, d) -> np.ndarray:
    """Code (uint8, 0..126) of e4m3 satfinite RNE(a / d) for exact a >= 0, d > 0."""
    return _rne_ratio(a, d, E4M3_POS).astype(np.uint8)


def e2m1_rne_ratio(a, d) -> np.ndarray:
    """Magnitude code (0..7) of e2m1 satfinite RNE(a / d) for exact a >= 0, d > 0."""
    return _rne_ratio(a, d, E2M1_MAG).astype(np.uint8)


# --------------------------------------------------------------- exact twins
def _rne_fraction(r: Fraction, values) -> int:
    """Index of RNE(r) among increasing exact ``values`` (ties to even index)."""
    if r >= values[-1]:
        return len(values) - 1
    i = max(j for j, v in enumerate(values) if v <= r)
    lo, hi = values[i], values[i + 1]
    mid = (lo + hi) / 2
    if r < mid:
        return i
    if r > mid:
        return i + 1
    return i if i % 2 == 0 else i + 1


_E4M3_POS_FRAC = E4M3_VALUE_FRAC[:127]


def e4m3_rne_fraction(r: Fraction) -> int:
    assert r >= 0
    return _rne_fraction(Fraction(r), _E4M3_POS_FRAC)


def e2m1_rne_fraction(r: Fraction) -> int:
    assert r >= 0
    return _rne_fraction(Fraction(r), E2M1_MAG_FRAC)
