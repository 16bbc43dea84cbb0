"""Pins for oracle.formats: e4m3 / e2m1 decoding and RNE rounding.

Independent references: torch's float8_e4m3fn conversions (a library
implementation of the same IEEE-style format), exhaustive nearest-value
search with exact rationals, and hand-listed midpoints.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F


def _torch_e4m3_decode_all():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_table_matches_torch():
    ref = _torch_e4m3_decode_all()
    ours = F.E4M3_VALUE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert F.E4M3_POS[-1] == 448.0 and F.E4M3_POS[1] == 2.0 ** -9


def test_e4m3_rne_matches_torch_cast():
    rng = np.random.default_rng(1)
    # random magnitudes over the whole range (normals and subnormals) + exact midpoints
    a = np.concatenate([
        rng.uniform(0, 448, 20000),
        np.exp2(rng.uniform(-12, 8.8, 20000)),
        (F.E4M3_POS[:-1] + F.E4M3_POS[1:]) / 2,
        F.E4M3_POS,
    ]).astype(np.float32)
    a = a[a <= 448]
    ours = F.e4m3_rne_ratio(a.astype(np.float64), 1.0)
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    assert F.e4m3_rne_ratio(np.array([448.0, 463.9, 464.0, 465, 1e30]), 1.0).tolist() == [126] * 5


@pytest.mark.parametrize("d", [3, 6])
def test_e4m3_ratio_bruteforce(d):
    """RNE(a/d) equals the exhaustive nearest e4m3 value (exact rationals, ties -> even code)."""
    # every a = e2m1 magnitude x e4m3 scale, the products requant rounds
    vals = sorted({Fraction(m) * s for m in F.E2M1_MAG_FRAC[1:] for s in F.E4M3_VALUE_FRAC[1:127]})
    pos = F.E4M3_VALUE_FRAC[:127]
    a64 = np.array([float(v) for v in vals])
    ours = F.e4m3_rne_ratio(a64, float(d))
    for a, got in zip(vals, ours):
        r = a / d
        best = None
        for c, v in enumerate(pos):
            dist = abs(r - v)
            if best is None or dist < best[0] or (dist == best[0] and c % 2 == 0):
                best = (dist, c)
        if r >= 448:
            best = (0, 126)
        assert got == best[1], (a, d, got, best)


def test_e4m3_subnormal_ties_of_s16():
    """The e4m3 ties of max|v|/3 (v = e2m1 x e4m3) all lie in the subnormal range."""
    ties = []
    for m in F.E2M1_MAG_FRAC[1:]:
        for s in F.E4M3_VALUE_FRAC[1:127]:
            r = m * s / 3
            for lo, hi in zip(F.E4M3_VALUE_FRAC[:126], F.E4M3_VALUE_FRAC[1:127]):
                if r == (lo + hi) / 2:
                    ties.append(r)
    assert len(ties) == 11
    assert all(r < Fraction(1, 64) for r in ties)       # below the smallest normal 2^-6
    # hand-worked: max|v| = 1.5 * 2^-9 -> /3 = 2^-10, the midpoint of 0 and 2^-9 -> even code 0
    assert F.e4m3_rne_ratio(np.array([1.5 * 2.0 ** -9]), 3.0)[0] == 0
    # 4.5 * 2^-9 -> 1.5 * 2^-9 = midpoint of codes 1 and 2 -> even code 2
    assert F.e4m3_rne_ratio(np.array([4.5 * 2.0 ** -9]), 3.0)[0] == 2


def test_e2m1_midpoints_hand_listed():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert F.e2m1_rne_ratio(mids, 1.0).tolist() == [0, 2, 2, 4, 4, 6, 6]
    eps = 1e-9
    assert F.e2m1_rne_ratio(mids + eps, 1.0).tolist() == [1, 2, 3, 4, 5, 6, 7]
    assert F.e2m1_rne_ratio(mids - eps, 1.0).tolist() == [0, 1, 2, 3, 4, 5, 6]
    assert F.e2m1_rne_ratio(np.array([0.0, 6.0, 6.5, 7.0, 1e9]), 1.0).tolist() == [0, 7, 7, 7, 7]
    assert F.e2m1_decode(np.arange(16)).tolist() == [0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6]


def test_fraction_twins_agree_with_fp64():
    rng = np.random.default_rng(2)
    s = F.E4M3_POS[rng.integers(1, 127, 3000)]
    m = F.E2M1_MAG[rng.integers(0, 8, 3000)]
    a = m * s + rng.integers(0, 8, 3000) * F.E4M3_POS[1] / 8     # exact dyadics
    for d in (3.0, 6.0, 0.34375):
        got = F.e4m3_rne_ratio(a, d)
        got2 = F.e2m1_rne_ratio(a, d * 64)
        for ai, g, g2 in zip(a[:600], got[:600], got2[:600]):
            assert g == F.e4m3_rne_fraction(Fraction(ai) / Fraction(d))
            assert g2 == F.e2m1_rne_fraction(Fraction(ai) / (Fraction(d) * 64))
