"""Pins for oracle.route and oracle.moe.

route: numpy's stable lexsort on (-logit, id), forced ties, NaN ordering,
weights summing to 1, the bucketing contract.
moe: a pure-Python loop brute force of the tiny layer with its own bit and
scale decoding (no oracle helper), linearity in the routing weights, and the
special cases "no delta table" == "gate all zero" and "k = 1, w = 1" == one
SwiGLU MLP.
"""
import math

import numpy as np
import pytest

import workloads as W
from oracle import moe, nvfp4, requant, route


# ------------------------------------------------------------------ route
def test_route_matches_lexsort():
    rng = np.random.default_rng(10)
    T, E, k = 37, 64, 6
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 5] = logits[:, 9]                # forced ties
    logits[3, :] = 0.5                          # a token with all-equal logits
    idx, w = route.route_topk(logits, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()
    assert idx[3].tolist() == list(range(k))
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)
    # weights are the full softmax renormalised over the chosen experts
    full = np.exp(logits.astype(np.float64) - logits.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


def test_route_nan_and_inf_ordering():
    logits = np.array([[np.nan, -np.inf, 1.0, 2.0]], dtype=np.float32)
    idx, w = route.route_topk(logits, 4)
    assert idx[0].tolist() == [3, 2, 1, 0]
    idx3, w3 = route.route_topk(logits, 3)       # NaN not selected: finite weights
    assert idx3[0].tolist() == [3, 2, 1]
    assert w3[0, 2] == 0.0 and abs(w3[0].sum() - 1.0) < 1e-15


def test_bucket_contract():
    rng = np.random.default_rng(11)
    T, E, k = 50, 16, 4
    idx, _ = route.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    counts, offsets, perm = route.bucket(idx, E)
    assert offsets[0] == 0 and offsets[E] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    assert sorted(perm.tolist()) == list(range(T * k))
    ref = np.argsort(idx.reshape(-1), kind="stable")
    assert np.array_equal(perm, ref)


# ------------------------------------------------------------------ forward
def _tiny_layer(cfg=W.CONFIGS["tiny"]):
    logits, xb, dset, gate = W.draw_layer_inputs(cfg)
    x = W.bf16_bits_to_f32(xb).astype(np.float64)
    fc = {1: {}, 2: {}}
    dfc = {1: {"codes": [], "s4": []}, 2: {"codes": [], "s4": []}}
    raw = {1: [], 2: []}
    for f in (1, 2):
        sg, mg, s16, sc2 = [], [], [], []
        for e in range(cfg.E):
            codes, s4, scale_2 = nvfp4.quantize(W.draw_weight(cfg, e, f))
            raw[f].append((codes, s4, scale_2))
            out = requant.requant_2bit(codes, s4)
            sg.append(out["sign"]); mg.append(out["mag"]); s16.append(out["s16"]); sc2.append(scale_2)
            if e in dset:
                dfc[f]["codes"].append(out["dcodes"]); dfc[f]["s4"].append(out["ds4"])
        fc[f] = dict(sign=np.stack(sg), mag=np.stack(mg), s16=np.stack(s16),
                     scale_2=np.array(sc2, dtype=np.float32))
        dfc[f] = {k_: np.stack(v) for k_, v in dfc[f].items()}
    idx, w = route.route_topk(logits, cfg.k)
    slot = W.delta_slot_table(cfg.E, dset)
    return cfg, x, idx, w, fc, dfc, slot, gate, raw


def _py_e4m3(b):
    e, m = (b >> 3) & 15, b & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)


def _py_w2(pl, e, r, K):
    """Row r of expert e's 2-bit matrix as a Python list (own decoder)."""
    row = []
    for k in range(K):
        word = int(pl["sign"][e, r, k // 32]); mword = int(pl["mag"][e, r, k // 32])
        s = (word >> (k % 32)) & 1
        m = (mword >> (k % 32)) & 1
        sc = _py_e4m3(int(pl["s16"][e, r, k // 16]))
        row.append((-1.0 if s else 1.0) * (3.0 if m else 1.0) * sc * float(pl["scale_2"][e]))
    return row


def _py_fp4(d, slot, r, K, scale_2):
    mags = [0, .5, 1, 1.5, 2, 3, 4, 6]
    row = []
    for k in range(K):
        byte = int(d["codes"][slot, r, k // 2])
        c = (byte >> 4) if k % 2 else (byte & 15)
        v = mags[c & 7] * (-1 if c & 8 else 1)
        row.append(v * _py_e4m3(int(d["s4"][slot, r, k // 16])) * float(scale_2))
    return row


def test_forward_bruteforce_tiny():
    cfg, x, idx, w, fc, dfc, slot, gate, _ = _tiny_layer()
    y = moe.moe_forward(x, idx, w, fc[1], fc[2], slot, dfc[1], dfc[2], gate)
    H, I = cfg.H, cfg.I
    cache = {}
    for t in range(cfg.T):
        yt = [0.0] * H
        for j in range(cfg.k):
            e = int(idx[t, j])
            wd = bool(gate[t]) and slot[e] >= 0
            key = (e, wd)
            if key not in cache:
                w1 = [_py_w2(fc[1], e, r, H) for r in range(2 * I)]
                w2 = [_py_w2(fc[2], e, r, I) for r in range(H)]
                if wd:
                    d1 = [_py_fp4(dfc[1], slot[e], r, H, fc[1]["scale_2"][e]) for r in range(2 * I)]
                    d2 = [_py_fp4(dfc[2], slot[e], r, I, fc[2]["scale_2"][e]) for r in range(H)]
                    w1 = [[a + b for a, b in zip(ra, rb)] for ra, rb in zip(w1, d1)]
                    w2 = [[a + b for a, b in zip(ra, rb)] for ra, rb in zip(w2, d2)]
                cache[key] = (w1, w2)
            w1, w2 = cache[key]
            xt = x[t].tolist()
            h = []
            for i in range(I):
                g = math.fsum(a * b for a, b in zip(w1[i], xt))
                u = math.fsum(a * b for a, b in zip(w1[I + i], xt))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for r in range(H):
                yt[r] += float(w[t, j]) * math.fsum(a * b for a, b in zip(w2[r], h))
        assert np.allclose(y[t], yt, rtol=1e-10, atol=1e-12)
    # the gated token really used the delta path (expert set {0, 3} is routed?)
    assert gate.tolist() == [0, 1, 0, 0]


def test_forward_linear_in_weights_and_delta_switches():
    cfg, x, idx, w, fc, dfc, slot, gate, _ = _tiny_layer()
    rng = np.random.default_rng(12)
    wa, wb = rng.random(w.shape), rng.random(w.shape)
    ya = moe.moe_forward(x, idx, wa, fc[1], fc[2], slot, dfc[1], dfc[2], gate)
    yb = moe.moe_forward(x, idx, wb, fc[1], fc[2], slot, dfc[1], dfc[2], gate)
    yab = moe.moe_forward(x, idx, wa + 2 * wb, fc[1], fc[2], slot, dfc[1], dfc[2], gate)
    assert np.allclose(yab, ya + 2 * yb, rtol=1e-12, atol=1e-14)
    y_none = moe.moe_forward(x, idx, w, fc[1], fc[2])
    y_gate0 = moe.moe_forward(x, idx, w, fc[1], fc[2], slot, dfc[1], dfc[2], np.zeros(cfg.T, np.uint8))
    y_noslot = moe.moe_forward(x, idx, w, fc[1], fc[2], np.full(cfg.E, -1, np.int32), dfc[1], dfc[2], gate)
    assert np.array_equal(y_none, y_gate0) and np.array_equal(y_none, y_noslot)


def test_forward_k1_is_one_mlp_and_delta_moves_toward_nvfp4():
    cfg, x, idx, w, fc, dfc, slot, gate, raw = _tiny_layer()
    e = 3                                     # an expert with a delta slot
    T = cfg.T
    idx1 = np.full((T, 1), e, dtype=np.int32)
    w1 = np.ones((T, 1))
    y = moe.moe_forward(x, idx1, w1, fc[1], fc[2])
    a1 = requant.dequant_2bit(fc[1]["sign"][e], fc[1]["mag"][e], fc[1]["s16"][e], fc[1]["scale_2"][e])
    a2 = requant.dequant_2bit(fc[2]["sign"][e], fc[2]["mag"][e], fc[2]["s16"][e], fc[2]["scale_2"][e])
    I = cfg.I
    g, u = x @ a1[:I].T, x @ a1[I:].T
    ref = (g / (1 + np.exp(-g)) * u) @ a2.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    # all gated with the delta: closer to the NVFP4 expert than the 2-bit one
    yd = moe.moe_forward(x, idx1, w1, fc[1], fc[2], slot, dfc[1], dfc[2], np.ones(T, np.uint8))
    n1 = nvfp4.dequantize(*raw[1][e]); n2 = nvfp4.dequantize(*raw[2][e])
    g, u = x @ n1[:I].T, x @ n1[I:].T
    yn = (g / (1 + np.exp(-g)) * u) @ n2.T
    assert np.linalg.norm(yd - yn) < 0.2 * np.linalg.norm(y - yn)


def test_forward_missing_experts_contribute_zero():
    """README "When the model doesn't fit at all": a routed expert that is not resident
    contributes zero (routing weights untouched).  Pinned against the full forward minus a
    textbook SwiGLU MLP (numpy matmuls on the dequantised weights) for every missing pair."""
    cfg, x, idx, w, fc, dfc, slot, gate, _ = _tiny_layer()
    I = cfg.I
    routed = sorted(set(int(e) for e in idx.ravel()))
    missing = set(routed[::2])
    resident = np.array([e not in missing for e in range(cfg.E)])
    y_full = moe.moe_forward(x, idx, w, fc[1], fc[2])
    y_res = moe.moe_forward(x, idx, w, fc[1], fc[2], resident=resident)
    expect = np.zeros_like(y_full)
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = int(idx[t, j])
            if e not in missing:
                continue
            a1 = requant.dequant_2bit(fc[1]["sign"][e], fc[1]["mag"][e], fc[1]["s16"][e], fc[1]["scale_2"][e])
            a2 = requant.dequant_2bit(fc[2]["sign"][e], fc[2]["mag"][e], fc[2]["s16"][e], fc[2]["scale_2"][e])
            g, u = a1[:I] @ x[t], a1[I:] @ x[t]
            expect[t] += w[t, j] * (a2 @ (g / (1 + np.exp(-g)) * u))
    assert missing and np.allclose(y_full - y_res, expect, rtol=1e-10, atol=1e-13)
    assert np.array_equal(moe.moe_forward(x, idx, w, fc[1], fc[2], resident=np.ones(cfg.E, bool)), y_full)
    assert not np.any(moe.moe_forward(x, idx, w, fc[1], fc[2], resident=np.zeros(cfg.E, bool)))


def test_gate_from_confidence_worked_example():
    """The gate: conf < tau strictly, NaN never gated; experts to promote = routed by a gated token
    and without a delta slot (each pair counted)."""
    from oracle import gate as ogate
    conf = np.array([0.9, 0.59, 0.6, np.nan, -np.inf, 0.2], dtype=np.float32)
    idx = np.array([[0, 1], [1, 2], [3, 0], [2, 3], [0, 3], [2, 1]], dtype=np.int32)
    slot = np.array([-1, 0, -1, 1], dtype=np.int32)        # experts 1 and 3 cached
    gate, need, n_gated, n_pairs = ogate.gate_from_confidence(conf, 0.6, idx, slot)
    assert gate.tolist() == [0, 1, 0, 0, 1, 1]              # 0.6 is not below 0.6; NaN never
    # gated tokens 1 (experts 1, 2), 4 (0, 3), 5 (2, 1): uncached 2, 0, 2
    assert need.tolist() == [True, False, True, False]
    assert (n_gated, n_pairs) == (3, 3)
    g2, need2, _, n2 = ogate.gate_from_confidence(conf, 0.6, idx, None)   # nothing cached
    assert g2.tolist() == gate.tolist() and need2.tolist() == [True, True, True, True] and n2 == 6
