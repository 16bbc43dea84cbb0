"""Sign-bias probe: per-block L2-optimal quantisation of weights to a 4-level integer codebook.

TEST INFRASTRUCTURE (see the package docstring).  README "Frontier MoE on consumer Blackwell
(SM120)", §"How it fits -- 2-bit experts at FP4 quality", bullet 1 ("the sign-bias finding"):
naive 2-bit quantisation fails through sign asymmetry, not error size -- the L2-optimal fit of
that codebook drops one sign's tail, so every expert carries a bias -- while a sign-symmetric
codebook at the same L2 error has a bias hundreds of times smaller.

The pages name neither the naive codebook nor the statistic.  Readings:
  * a codebook is 4 ascending integer levels L; the naive one is the two's-complement int2 grid
    {-2, -1, 0, 1}, whose range reaches one sign's tail only (symmetric ones: {-3, -1, 1, 3}, this
    library's, and the pages' {-4, -1, 1, 4});
  * each block of 16 consecutive weights along K (the 2-bit planes' scale block) gets the scale
    s > 0 minimising sum_i (w_i - s L[a_i])^2 with a_i the nearest level to w_i / s;
  * per matrix the probe reports sum W, sum W^2, the bias sum (Q - W) and the error sum (Q - W)^2.

The exact optimum.  For s > 0 the nearest-level assignment is monotone in w, so the optimum is
among the monotone assignments of the sorted block: c1 smallest weights -> L0, the next c2 - c1
-> L1, c3 - c2 -> L2, the rest -> L3, for 0 <= c1 <= c2 <= c3 <= 16 (969 candidates).  For one
assignment the best scale is s = Nc / Dc with Nc = sum a_i w_i and Dc = sum a_i^2, leaving the
error sum w^2 - Nc^2 / Dc, so the best candidate maximises Nc^2 / Dc among those with Nc > 0
(s > 0); if none has Nc > 0 the block quantises to 0.  Where several candidates reach the same
maximum exactly, the first in the order c1, then c2, then c3 ascending is taken.

Decision arithmetic.  The argmax decides an integer (the assignment), so it is taken exactly:
the block's fp32 weights are integers times one power of two, 2^E, so every prefix sum P and
every Nc = (L0 - L1) P[c1] + (L1 - L2) P[c2] + (L2 - L3) P[c3] + L3 P[16] is an exact integer
times 2^E (int64 when the block's magnitudes span at most 24 binades, Python integers
otherwise), and Dc is an integer.  Scores are ranked in fp64 and every candidate within a
relative 1e-9 of the top fp64 score is compared exactly, Nc_a^2 Dc_b against Nc_b^2 Dc_a in
integers.  The chosen block's sums are then evaluated in fp64: Nc and sum a_i from the counts
and the fp64 sums of the four groups, s = Nc / Dc, bias = s sum a - sum w, error = sum w^2 -
Nc^2 / Dc.  Each block also reports its decision margin (the relative gap between the best score
and the best score of a candidate with a different, exactly smaller score) and its Nc, so that
an implementation that ranks the candidates in lower precision can be held to the exact choice
wherever the margin exceeds its rounding error.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
NAIVE_INT2 = (-2, -1, 0, 1)
SYMMETRIC_13 = (-3, -1, 1, 3)
SYMMETRIC_14 = (-4, -1, 1, 4)


def _candidates(B: int):
    """All (c1, c2, c3) with 0 <= c1 <= c2 <= c3 <= B, in the search order."""
    return [(c1, c2, c3) for c1 in range(B + 1) for c2 in range(c1, B + 1) for c3 in range(c2, B + 1)]


_CAND_CACHE = {}


def _cand_arrays(B: int):
    if B not in _CAND_CACHE:
        c = np.array(_candidates(B), dtype=np.int64)
        _CAND_CACHE[B] = (c[:, 0], c[:, 1], c[:, 2])
    return _CAND_CACHE[B]


def _block_integers(ws: np.ndarray):
    """Sorted fp32 blocks [nb, B] -> (n [nb, B] integers as Python-int object array or int64, E [nb])
    with ws = n * 2^E exactly; int64 where every block spans at most 24 binades."""
    ws = np.asarray(ws, dtype=np.float32)
    a = np.abs(ws.astype(np.float64))
    nz = a > 0
    big = np.where(nz, a, 0.0).max(axis=1)
    small = np.where(nz, a, np.inf).min(axis=1)
    e_small = np.where(np.isfinite(small), np.floor(np.log2(np.where(np.isfinite(small), small, 1.0))), 0.0)
    e_big = np.where(big > 0, np.floor(np.log2(np.where(big > 0, big, 1.0))), 0.0)
    E = np.maximum(e_small - 23, -149).astype(np.int64)            # ulp exponent of the smallest |w|
    spread = (e_big - e_small).astype(np.int64)
    n = ws.astype(np.float64) * np.ldexp(1.0, -E)[:, None]          # exact integers (fp64 holds 2^53)
    ok = spread <= 24
    return n, E, ok


def _exact_int(x) -> int:
    return int(x)


def _decide(n_rows, levels):
    """Exact argmax over the candidates for integer blocks n_rows [m, B] (Python ints or int64 in
    float64 storage).  Returns (cut [m, 3] (-1 = none), margin [m], nbest [m] float)."""
    m, B = n_rows.shape
    L0, L1, L2, L3 = (int(v) for v in levels)
    c1, c2, c3 = _cand_arrays(B)
    D = ((L0 * L0 - L1 * L1) * c1 + (L1 * L1 - L2 * L2) * c2 + (L2 * L2 - L3 * L3) * c3
         + B * L3 * L3).astype(np.int64)
    A, Bc, C = L0 - L1, L1 - L2, L2 - L3
    cut = np.full((m, 3), -1, dtype=np.int64)
    margin = np.zeros(m)
    nbest = np.zeros(m)
    for r in range(m):
        P = [0]
        for j in range(B):
            P.append(P[-1] + _exact_int(n_rows[r, j]))
        Pa = np.array(P, dtype=object)
        N = A * Pa[c1] + Bc * Pa[c2] + C * Pa[c3] + L3 * Pa[B]          # exact (Python ints)
        Nf = N.astype(np.float64)
        pos = Nf > 0
        if not pos.any():
            continue
        with np.errstate(divide="ignore", invalid="ignore"):
            score = np.where(pos, Nf * Nf / D, -1.0)
        top = score.max()
        near = np.flatnonzero(score >= top * (1.0 - 1e-9))
        best = int(near[0])
        for i in near[1:]:                                             # exact: N_i^2 D_b > N_b^2 D_i
            i = int(i)
            if N[i] * N[i] * int(D[best]) > N[best] * N[best] * int(D[i]):
                best = i
        # the best score of any other candidate (an exact tie gives margin 0)
        others = np.delete(score, best)
        second = others.max() if others.size else -1.0
        margin[r] = (score[best] - second) / score[best] if second > 0 else 1.0
        cut[r] = (c1[best], c2[best], c3[best])
        nbest[r] = float(N[best])
    return cut, margin, nbest


def _decide_fast(n, levels):
    """Vectorised twin of _decide for int64-range blocks: exact integer N in int64, fp64 ranking,
    exact comparison (Python ints) of the candidates that come within 1e-9 of the top."""
    nb, B = n.shape
    L0, L1, L2, L3 = (int(v) for v in levels)
    c1, c2, c3 = _cand_arrays(B)
    D = ((L0 * L0 - L1 * L1) * c1 + (L1 * L1 - L2 * L2) * c2 + (L2 * L2 - L3 * L3) * c3
         + B * L3 * L3).astype(np.int64)
    ni = n.astype(np.int64)
    P = np.zeros((nb, B + 1), dtype=np.int64)
    P[:, 1:] = np.cumsum(ni, axis=1)
    N = (L0 - L1) * P[:, c1] + (L1 - L2) * P[:, c2] + (L2 - L3) * P[:, c3] + L3 * P[:, B:B + 1]   # [nb, 969]
    Nf = N.astype(np.float64)
    pos = Nf > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        score = np.where(pos, Nf * Nf / D[None, :], -1.0)
    top = score.max(axis=1)
    cut = np.full((nb, 3), -1, dtype=np.int64)
    margin = np.zeros(nb)
    nbest = np.zeros(nb)
    has = top > 0
    near = score >= (top * (1.0 - 1e-9))[:, None]
    first = np.argmax(near, axis=1)
    multi = near.sum(axis=1) > 1
    best = first.copy()
    for r in np.flatnonzero(multi & has):
        cand = np.flatnonzero(near[r])
        b = int(cand[0])
        for i in cand[1:]:
            i = int(i)
            if int(N[r, i]) ** 2 * int(D[b]) > int(N[r, b]) ** 2 * int(D[i]):
                b = i
        best[r] = b
    sb_ = score[np.arange(nb), best]
    # the best score of any other candidate (an exact tie gives margin 0)
    rest = score.copy()
    rest[np.arange(nb), best] = -1.0
    second = rest.max(axis=1)
    margin = np.where(has, np.where(second > 0, (sb_ - second) / np.where(sb_ > 0, sb_, 1.0), 1.0), 0.0)
    cut[has] = np.stack([c1[best], c2[best], c3[best]], axis=1)[has]
    nbest[has] = Nf[np.arange(nb), best][has]
    return cut, margin, nbest


def probe_blocks(w: np.ndarray, levels, block: int = BLOCK):
    """One [N, K] matrix -> (per-block sums [N, K/block, 4] (sum W, sum W^2, sum (Q - W),
    sum (Q - W)^2), decision margin [N, K/block], Nc of the choice in units of 2^E times 2^E
    (fp64) [N, K/block], sum |W| [N, K/block])."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % block == 0
    ws = np.sort(w.reshape(-1, block), axis=1)
    nb = ws.shape[0]
    L0, L1, L2, L3 = (int(v) for v in levels)
    n, E, ok = _block_integers(ws)
    cut = np.full((nb, 3), -1, dtype=np.int64)
    margin = np.zeros(nb)
    nbest = np.zeros(nb)
    if ok.any():
        c, mg, nbv = _decide_fast(n[ok], levels)
        cut[ok], margin[ok], nbest[ok] = c, mg, nbv
    if (~ok).any():
        from fractions import Fraction
        rows = np.flatnonzero(~ok)
        for r in rows:                     # wide blocks: exact Python integers
            ints = np.array([int(Fraction(float(x)) / Fraction(2) ** int(E[r])) for x in ws[r]], dtype=object)
            c, mg, nbv = _decide(ints[None, :], levels)
            cut[r], margin[r], nbest[r] = c[0], mg[0], nbv[0]
    wd = ws.astype(np.float64)
    sw, sw2 = wd.sum(axis=1), (wd * wd).sum(axis=1)
    idx = np.arange(block)[None, :]
    a = np.where(idx < cut[:, 0:1], L0, np.where(idx < cut[:, 1:2], L1,
                                                 np.where(idx < cut[:, 2:3], L2, L3))).astype(np.float64)
    nc, dc = (a * wd).sum(axis=1), (a * a).sum(axis=1)
    found = cut[:, 0] >= 0
    with np.errstate(divide="ignore", invalid="ignore"):
        bias = np.where(found, nc / dc * a.sum(axis=1) - sw, -sw)
        err = np.where(found, sw2 - nc * nc / dc, sw2)
    per_block = np.stack([sw, sw2, bias, err], axis=1).reshape(N, K // block, 4)
    return (per_block, margin.reshape(N, K // block), (nbest * np.ldexp(1.0, E)).reshape(N, K // block),
            np.abs(wd).sum(axis=1).reshape(N, K // block))


def best_assignment(ws: np.ndarray, levels):
    """(c1, c2, c3) of the exact best candidate for one sorted fp32 block, or None when no
    candidate has Nc > 0."""
    ws = np.sort(np.asarray(ws, dtype=np.float32))
    from fractions import Fraction
    den = max(Fraction(float(x)).denominator for x in ws)      # a power of two: x den is an integer
    ints = np.array([int(Fraction(float(x)) * den) for x in ws], dtype=object)
    cut, _, _ = _decide(ints[None, :], levels)
    return None if cut[0, 0] < 0 else tuple(int(v) for v in cut[0])


def block_sums(w: np.ndarray, levels) -> tuple:
    """(sum w, sum w^2, bias sum (Q - w), error sum (Q - w)^2) of one block, fp64 (the exact choice
    made with Python integers throughout)."""
    w = np.asarray(w, dtype=np.float32)
    B = w.shape[0]
    ws = np.sort(w)
    wd = ws.astype(np.float64)
    sw, sw2 = float(wd.sum()), float((wd * wd).sum())
    cand = best_assignment(ws, levels)
    if cand is None:
        return sw, sw2, -sw, sw2
    c1, c2, c3 = cand
    cuts = (0, c1, c2, c3, B)
    a = np.concatenate([np.full(cuts[j + 1] - cuts[j], float(levels[j])) for j in range(4)])
    nc = float((a * wd).sum())
    dc = float((a * a).sum())
    s = nc / dc
    return sw, sw2, s * float(a.sum()) - sw, sw2 - nc * nc / dc


def probe(w: np.ndarray, levels, block: int = BLOCK) -> np.ndarray:
    """One [N, K] matrix -> [N, 4] per-row sums (sum W, sum W^2, sum (Q - W), sum (Q - W)^2)."""
    return probe_blocks(w, levels, block)[0].sum(axis=1)


def statistics(sums: np.ndarray, n_weights: int) -> dict:
    """Statistics of one matrix from its summed (sum W, sum W^2, bias sum, error sum):
    bias = mean(Q - W) / rms(W) and rel_rms = ||Q - W|| / ||W||."""
    sw, sw2, sb, se = (float(x) for x in sums)
    rms = np.sqrt(sw2 / n_weights)
    return {"bias": sb / n_weights / rms, "rel_rms": float(np.sqrt(se / sw2))}
