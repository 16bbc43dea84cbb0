"""Router top-k with renormalised softmax, and the token bucketing by expert.

Routing step of the MoE layer (README "Frontier MoE on consumer Blackwell
(SM120)", §"How it fits"; the DeepSeek-V4.1 table on the airanks page, row
"MoE at decode", describes the router -> FC1 launch chain this replaces):

  selection  per token, the k experts with the largest logits, in order of
             decreasing logit; equal logits go to the lower expert id; NaN
             ranks below -inf.
  weights    w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k
             selected logits (= the full softmax renormalised over the top-k).
  bucketing  counts[e] = number of (token, slot) pairs routed to e;
             offsets = exclusive prefix sum, offsets[E] = T*k;
             perm lists the pair ids p = t*k + j grouped by expert in
             increasing e, and by increasing p within an expert.
"""
from __future__ import annotations

import math

import numpy as np


def _rank_key(e: int, logit: float):
    if math.isnan(logit):
        return (1, 0.0, e)
    return (0, -logit, e)


def route_topk(logits: np.ndarray, k: int):
    """logits [T, E] fp32 -> (idx [T, k] int32, w [T, k] fp64)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    idx = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        row = [float(v) for v in logits[t]]
        chosen = sorted(range(E), key=lambda e: _rank_key(e, row[e]))[:k]
        lmax = row[chosen[0]]
        ex = [math.exp(row[e] - lmax) for e in chosen]
        s = math.fsum(ex)
        idx[t] = chosen
        w[t] = [v / s for v in ex]
    return idx, w


def bucket(idx: np.ndarray, E: int):
    """idx [T, k] -> (counts [E], offsets [E+1], perm [T*k]) as int32."""
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        counts[int(e)] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    perm = np.zeros(T * k, dtype=np.int64)
    fill = offsets[:-1].copy()
    for p in range(T * k):                 # increasing p keeps each bucket stable
        e = int(idx.reshape(-1)[p])
        perm[fill[e]] = p
        fill[e] += 1
    return counts.astype(np.int32), offsets.astype(np.int32), perm.astype(np.int32)
