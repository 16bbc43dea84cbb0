"""Pins of the sign-bias probe oracle (oracle/signbias.py) against definitions it does not use:
exhaustive assignments compared exactly in rational arithmetic, a direct scan over scales with
nearest-level rounding, exact fits, scale and sign symmetries, and the pages' qualitative
finding on synthetic weights."""
import itertools

import numpy as np
import pytest

from oracle import signbias as sb

CODEBOOKS = [sb.NAIVE_INT2, sb.SYMMETRIC_13, sb.SYMMETRIC_14]


def _nearest_error(w, levels, s):
    """sum (w - s L[nearest])^2 and sum (Q - w) at scale s, by direct rounding (fp64)."""
    L = np.asarray(levels, dtype=np.float64)
    q = L[np.argmin(np.abs(w[:, None] / s - L[None, :]), axis=1)] * s
    return float(((q - w) ** 2).sum()), float((q - w).sum())


def _exact_error(w, a):
    """sum w^2 - (sum a w)^2 / sum a^2 in exact rationals (w fp32, a integer levels)."""
    from fractions import Fraction
    wf = [Fraction(float(x)) for x in w]
    nc = sum(int(ai) * wi for ai, wi in zip(a, wf))
    dc = sum(int(ai) * int(ai) for ai in a)
    sw2 = sum(x * x for x in wf)
    return sw2 - nc * nc / dc if (dc > 0 and nc > 0) else sw2


def _chosen_levels(ws, levels):
    cand = sb.best_assignment(ws, levels)
    if cand is None:
        return None
    cuts = (0,) + cand + (len(ws),)
    return [levels[j] for j in range(4) for _ in range(cuts[j + 1] - cuts[j])]


@pytest.mark.parametrize("levels", CODEBOOKS)
def test_search_equals_exhaustive_assignments(levels):
    """On blocks of 6 weights the exact monotone search reaches the minimum of
    sum w^2 - Nc^2/Dc over all 4^6 assignments with Nc > 0 (sum w^2 when none has) exactly, in
    rational arithmetic: the L2 optimum over every (assignment, scale > 0) pair.  Blocks include
    one-signed ones and blocks spanning 60 binades (the exact path beyond int64)."""
    rng = np.random.default_rng(41)
    combos = list(itertools.product(range(4), repeat=6))
    for it in range(40):
        w = rng.standard_normal(6).astype(np.float32)
        if rng.random() < 0.3:
            w = np.abs(w) * (1 if rng.random() < 0.5 else -1)            # one-signed blocks
        if it % 7 == 3:
            w[:2] *= np.float32(1e-18)                                     # wide magnitude span
        ws = np.sort(w)
        best = min(_exact_error(ws, [levels[c] for c in combo]) for combo in combos)
        a = _chosen_levels(ws, levels)
        got = _exact_error(ws, a) if a is not None else _exact_error(ws, [0] * 6)
        assert got == best, (it, float(got), float(best))


@pytest.mark.parametrize("levels", CODEBOOKS)
def test_vectorised_choice_equals_exact_scalar_choice(levels):
    """The vectorised search (int64 integers, fp64 ranking, exact comparison of near-top
    candidates) takes the same assignment as the scalar one in Python integers throughout, on
    blocks of 16 with repeated values, exact ties and one-signed blocks; an exact tie reports
    margin 0."""
    rng = np.random.default_rng(47)
    w = (rng.standard_t(4, (6, 64)) * 0.02).astype(np.float32)
    w[0, :16] = np.float32(0.01)                                           # all equal
    w[1, 16:32] = np.abs(w[1, 16:32])
    w[2, :16] = np.repeat(w[2, :4], 4)
    w[3, :16] = np.float32(0.25) * np.asarray(levels, np.float32)[np.arange(16) % 4]
    per_block, margin, _, _ = sb.probe_blocks(w, levels)
    for n in range(w.shape[0]):
        for b in range(4):
            ref = sb.block_sums(w[n, 16 * b:16 * b + 16], levels)
            assert np.allclose(per_block[n, b], ref, rtol=1e-13, atol=1e-18), (n, b)
    # two distinct weights, 8 each: the cut between them can sit at two places with equal scores
    # for {-1, 1}-symmetric pairs of levels -> at least one exact tie somewhere in such blocks
    assert (margin >= 0).all() and (margin <= 1).all()


@pytest.mark.parametrize("levels", CODEBOOKS)
def test_search_beats_every_scale_of_a_direct_scan(levels):
    """Blocks of 16: the error is at most the nearest-level error at every scanned scale and at
    least the scan's minimum less its resolution; the bias matches the scan's best scale."""
    rng = np.random.default_rng(42)
    for _ in range(12):
        w = (rng.standard_t(4, 16) * 0.02).astype(np.float32)
        wd = w.astype(np.float64)
        sw, sw2, bias, err = sb.block_sums(w, levels)
        smax = np.abs(wd).max() / 0.4
        scales = np.linspace(smax / 20000, smax, 20000)
        scan = np.array([_nearest_error(wd, levels, s) for s in scales])
        assert err <= scan[:, 0].min() + 1e-15
        assert err >= scan[:, 0].min() - 1e-3 * sw2
        assert bias == pytest.approx(scan[np.argmin(scan[:, 0]), 1], abs=0.05 * np.sqrt(sw2))


@pytest.mark.parametrize("levels", CODEBOOKS)
def test_exact_fit_has_no_error_and_no_bias(levels):
    rng = np.random.default_rng(43)
    a = np.asarray(levels, dtype=np.float64)[rng.permutation(np.arange(16) % 4)]
    w = (0.375 * a).astype(np.float32)
    sw, sw2, bias, err = sb.block_sums(w, levels)
    assert abs(err) <= 1e-12 * sw2 and abs(bias) <= 1e-12 * np.sqrt(sw2)


@pytest.mark.parametrize("levels", CODEBOOKS)
def test_power_of_two_scale_and_sign(levels):
    """Doubling W doubles the sums of W and of Q - W and quadruples the squares, exactly; for a
    sign-symmetric codebook negating W negates the two signed sums and keeps the squares."""
    rng = np.random.default_rng(44)
    w = (rng.standard_t(4, (8, 64)) * 0.02).astype(np.float32)
    a = sb.probe(w, levels)
    b = sb.probe(w * np.float32(2), levels)
    assert np.array_equal(b, a * np.array([2, 4, 2, 4]))
    if levels[0] == -levels[3] and levels[1] == -levels[2]:
        c = sb.probe(-w, levels)
        assert np.allclose(c, a * np.array([-1, 1, -1, 1]), rtol=1e-12, atol=1e-18)


def test_zero_block_and_vectorised_equals_scalar():
    z = sb.probe(np.zeros((2, 32), np.float32), sb.NAIVE_INT2)
    assert not z.any()
    rng = np.random.default_rng(45)
    w = (rng.standard_t(4, (3, 48)) * 0.02).astype(np.float32)
    w[0, :16] = np.abs(w[0, :16])
    w[1, 16:32] = -np.abs(w[1, 16:32])
    for levels in CODEBOOKS:
        v = sb.probe(w, levels)
        ref = np.array([[sum(x) for x in zip(*[sb.block_sums(w[n, 16 * b:16 * b + 16], levels)
                                               for b in range(3)])] for n in range(3)])
        assert np.allclose(v, ref, rtol=1e-13, atol=1e-18)


def test_the_pages_finding_on_synthetic_weights():
    """README "How it fits", bullet 1: the naive codebook's optimal fit carries a bias of one sign
    on (nearly) every tensor, a symmetric one a far smaller bias at a similar L2 error."""
    rng = np.random.default_rng(46)
    stats = {levels: [] for levels in CODEBOOKS}
    for m in range(6):
        w = (rng.standard_t(4, (32, 512)) * 0.02 / np.sqrt(2)).astype(np.float32)
        for levels in CODEBOOKS:
            stats[levels].append(sb.statistics(sb.probe(w, levels).sum(0), w.size))
    naive = stats[sb.NAIVE_INT2]
    assert all(s["bias"] < -0.01 for s in naive)
    for levels in (sb.SYMMETRIC_13, sb.SYMMETRIC_14):
        mean_abs = np.mean([abs(s["bias"]) for s in stats[levels]])
        assert mean_abs * 10 < np.mean([abs(s["bias"]) for s in naive])
        for s, n in zip(stats[levels], naive):
            assert 0.8 < s["rel_rms"] / n["rel_rms"] < 1.2
