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
(s > 0); if none has Nc > 0 the block quantises to 0.

Decision precision.  The argmax decides an integer (the assignment), so it is taken in fp32 with
one fixed operation order, which the GPU kernel follows too:
  P[0] = 0, P[j + 1] = fl(P[j] + w_sorted[j])                      (fp32 prefix sums)
  N = fl(fl(fl(fl(A P[c1]) + fl(B P[c2])) + fl(C P[c3])) + fl(Dl P[16]))
      with A = L0 - L1, B = L1 - L2, C = L2 - L3, Dl = L3          (integers)
  D = (L0^2 - L1^2) c1 + (L1^2 - L2^2) c2 + (L2^2 - L3^2) c3 + 16 L3^2  (exact)
  candidates in the order c1, then c2, then c3 ascending; one replaces the best when N > 0 and
  fl(fl(N N) Dbest) > fl(NNbest D)                               (first maximum wins)
The chosen block's sums are then evaluated in fp64: Nc and sum a_i from the counts and the fp64
sums of the four groups, s = Nc / Dc, bias = s sum a - sum w, error = sum w^2 - Nc^2 / Dc.
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


def best_assignment(ws: np.ndarray, levels) -> tuple:
    """The search on one sorted block ws (fp32, ascending): (c1, c2, c3) of the best candidate, or
    None when no candidate has N > 0."""
    ws = np.asarray(ws, dtype=np.float32)
    B = ws.shape[0]
    L0, L1, L2, L3 = (int(v) for v in levels)
    f32 = np.float32
    P = [f32(0)]
    for j in range(B):
        P.append(f32(P[-1] + ws[j]))
    A, Bc, C, Dl = f32(L0 - L1), f32(L1 - L2), f32(L2 - L3), f32(L3)
    best, nn_best, d_best = None, f32(0), f32(1)
    for c1, c2, c3 in _candidates(B):
        n = f32(f32(f32(f32(A * P[c1]) + f32(Bc * P[c2])) + f32(C * P[c3])) + f32(Dl * P[B]))
        d = f32((L0 * L0 - L1 * L1) * c1 + (L1 * L1 - L2 * L2) * c2 + (L2 * L2 - L3 * L3) * c3 + B * L3 * L3)
        if n > 0:
            nn = f32(n * n)
            if f32(nn * d_best) > f32(nn_best * d):
                best, nn_best, d_best = (c1, c2, c3), nn, d
    return best


def block_sums(w: np.ndarray, levels) -> tuple:
    """(sum w, sum w^2, bias sum (Q - w), error sum (Q - w)^2) of one block, fp64."""
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
    """One [N, K] matrix -> [N, 4] per-row sums (sum W, sum W^2, sum (Q - W), sum (Q - W)^2).
    The same search as best_assignment / block_sums, run on all blocks at once (every fp32
    operation is the same elementwise operation on arrays)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % block == 0
    ws = np.sort(w.reshape(-1, block), axis=1)
    nb = ws.shape[0]
    L0, L1, L2, L3 = (int(v) for v in levels)
    f32 = np.float32
    P = np.zeros((nb, block + 1), dtype=np.float32)
    for j in range(block):
        P[:, j + 1] = P[:, j] + ws[:, j]
    A, Bc, C, Dl = f32(L0 - L1), f32(L1 - L2), f32(L2 - L3), f32(L3)
    tail = Dl * P[:, block]
    cut = np.full((nb, 3), -1, dtype=np.int64)
    nn_best = np.zeros(nb, dtype=np.float32)
    d_best = np.ones(nb, dtype=np.float32)
    for c1, c2, c3 in _candidates(block):
        n = ((A * P[:, c1] + Bc * P[:, c2]) + C * P[:, c3]) + tail
        d = f32((L0 * L0 - L1 * L1) * c1 + (L1 * L1 - L2 * L2) * c2 + (L2 * L2 - L3 * L3) * c3
                + block * L3 * L3)
        nn = n * n
        upd = (n > 0) & (nn * d_best > nn_best * d)
        cut[upd] = (c1, c2, c3)
        nn_best[upd] = nn[upd]
        d_best[upd] = d
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
    per_block = np.stack([sw, sw2, bias, err], axis=1)
    return per_block.reshape(N, K // block, 4).sum(axis=1)


def statistics(sums: np.ndarray, n_weights: int) -> dict:
    """Statistics of one matrix from its summed (sum W, sum W^2, bias sum, error sum):
    bias = mean(Q - W) / rms(W) and rel_rms = ||Q - W|| / ||W||."""
    sw, sw2, sb, se = (float(x) for x in sums)
    rms = np.sqrt(sw2 / n_weights)
    return {"bias": sb / n_weights / rms, "rel_rms": float(np.sqrt(se / sw2))}
