"""The MoE expert-layer forward over 2-bit planes with the NVFP4 delta.

README "Frontier MoE on consumer Blackwell (SM120)", §"How it fits -- 2-bit
experts at FP4 quality", bullet 2: decode streams the 2-bit experts; a delta
cache keeps hot experts at FP4 and a confidence gate re-runs low-confidence
tokens at FP4.  As a layer computation:

  y_t = sum_j w_tj * FFN_{e_tj}(x_t)
  FFN_e(x) = W2_e ( SiLU(Wg_e x) * (Wu_e x) ),   SiLU(z) = z / (1 + e^-z)

FC1 = [Wg; Wu] is [2I, H] (gate rows first, then up rows), FC2 = W2 is
[H, I].  Each weight matrix is the dequantised 2-bit plane set
q * s16 * scale_2, and it becomes W_2bit + Delta exactly for the pairs whose
token is flagged by the gate mask and whose expert holds a delta-pool slot
(the delta is the NVFP4 residual on the same scale_2).  No SwiGLU clamp is
applied (the airanks page's audit note mentions one for a specific
checkpoint; this layer is plain SiLU*mul).

Everything is fp64: activations enter as their exact bf16 values and every
weight is dequantised exactly.  The k=1 and single-MLP special cases and a
pure-Python brute force on the tiny layer pin this function in the tests.
"""
from __future__ import annotations

import numpy as np

from .nvfp4 import dequantize_units
from .requant import dequant_2bit_units


def silu(z):
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_weights(e, fc1, fc2, delta_slot=None, dfc1=None, dfc2=None, with_delta=False):
    """fp64 (W1 [2I, H], W2 [H, I]) of expert e, with the delta added if asked."""
    w1 = dequant_2bit_units(fc1["sign"][e], fc1["mag"][e], fc1["s16"][e])
    w2 = dequant_2bit_units(fc2["sign"][e], fc2["mag"][e], fc2["s16"][e])
    if with_delta:
        s = int(delta_slot[e])
        assert s >= 0
        w1 = w1 + dequantize_units(dfc1["codes"][s], dfc1["s4"][s])
        w2 = w2 + dequantize_units(dfc2["codes"][s], dfc2["s4"][s])
    return w1 * np.float64(fc1["scale_2"][e]), w2 * np.float64(fc2["scale_2"][e])


def ffn(x: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """SwiGLU expert MLP for x [n, H] -> [n, H] in fp64."""
    I = w1.shape[0] // 2
    g = x @ w1[:I].T
    u = x @ w1[I:].T
    return (silu(g) * u) @ w2.T


def moe_forward(x, idx, w, fc1, fc2, delta_slot=None, dfc1=None, dfc2=None, gate=None,
                tokens=None, resident=None):
    """y [T, H] fp64.  ``x`` holds fp64 activation values (exact bf16 values).

    ``tokens`` optionally restricts the computation to a subset of token ids
    (rows of the returned array outside the subset are zero); used to check
    sampled outputs of full-size layers.

    ``resident`` optionally marks which experts are resident on the GPU (bool
    [E]); a pair routed to an expert that is not contributes zero (README
    "Frontier MoE on consumer Blackwell (SM120)", "When the model doesn't fit at
    all -- the GPU as an expert cache": the missing expert's contribution is
    zeroed and counted, the routing weights are left as they are).
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    k = idx.shape[1]
    y = np.zeros((T, H), dtype=np.float64)
    tok_set = range(T) if tokens is None else sorted(set(int(t) for t in tokens))
    use_delta = delta_slot is not None and gate is not None
    pairs = {}                                  # (expert, with_delta) -> [(t, j)]
    for t in tok_set:
        for j in range(k):
            e = int(idx[t, j])
            if resident is not None and not resident[e]:
                continue
            wd = bool(use_delta and gate[t] and delta_slot[e] >= 0)
            pairs.setdefault((e, wd), []).append((t, j))
    for (e, wd), plist in sorted(pairs.items()):
        w1, w2 = expert_weights(e, fc1, fc2, delta_slot, dfc1, dfc2, with_delta=wd)
        ts = np.array([t for t, _ in plist])
        js = np.array([j for _, j in plist])
        o = ffn(x[ts], w1, w2)
        for r in range(len(plist)):             # fixed order, one pair at a time
            y[ts[r]] += np.float64(w[ts[r], js[r]]) * o[r]
    return y
