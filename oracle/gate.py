"""The confidence gate's producer (oracle; test infrastructure only).

README "Frontier MoE on consumer Blackwell (SM120)", §"How it fits -- 2-bit
experts at FP4 quality" (the FP4 tier): a confidence gate re-runs low-confidence
steps at FP4, promoting the step's routed experts into the delta cache before
the replay.  The pages leave the confidence undefined; the reading used here is
one value per token given by the caller, and token t is gated when
conf[t] < tau (strictly; NaN is never below tau).  For the replay the caller
must promote every expert that a gated token routes to and that holds no delta
slot.
"""
from __future__ import annotations

import numpy as np


def gate_from_confidence(conf, tau, idx, delta_slot=None):
    """Returns (gate u8 [T], need bool [E], n_gated, n_need_pairs) for conf [T], idx [T, k].

    ``E`` is taken from ``delta_slot`` ([E], -1 = not cached; None = nothing cached) or, without
    one, from the largest routed expert id + 1."""
    conf = np.asarray(conf, dtype=np.float32)
    idx = np.asarray(idx)
    T, k = idx.shape
    E = len(delta_slot) if delta_slot is not None else int(idx.max()) + 1
    gate = np.zeros(T, dtype=np.uint8)
    need = np.zeros(E, dtype=bool)
    n_gated = n_pairs = 0
    for t in range(T):
        if not (conf[t] < np.float32(tau)):
            continue
        gate[t] = 1
        n_gated += 1
        for j in range(k):
            e = int(idx[t, j])
            if delta_slot is None or delta_slot[e] < 0:
                need[e] = True
                n_pairs += 1
    return gate, need, n_gated, n_pairs
