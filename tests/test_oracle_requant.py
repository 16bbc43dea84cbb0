"""Pins for oracle.nvfp4 (input quantiser) and oracle.requant (2-bit planes + delta).

Independent references: hand-worked examples under tests/golden/, exhaustive
nearest-level search with exact rationals, and the invariants the method
states (never-zero code, sign symmetry, delta reconstruction bound).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import nvfp4, requant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _pack_codes(codes):
    codes = np.asarray(codes, dtype=np.uint8).reshape(1, -1)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_worked_example():
    g = _load("nvfp4_worked_example.json")
    w = np.array(g["w"], dtype=np.float32).reshape(1, -1)
    packed, s4, scale_2 = nvfp4.quantize(w)
    assert float(scale_2) == g["expect_scale_2"]
    assert s4.reshape(-1).tolist() == g["expect_s4_codes"]
    assert nvfp4.unpack_codes(packed).reshape(-1).tolist() == g["expect_codes"]


def _brute_nearest(r: Fraction, levels):
    """Index of the level nearest r; ties -> even index; saturate at the top."""
    if r >= levels[-1]:
        return len(levels) - 1
    best = None
    for i, v in enumerate(levels):
        d = abs(r - v)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_nvfp4_bruteforce_small():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((3, 32)) * np.exp2(rng.integers(-8, 4, (3, 1)))).astype(np.float32)
    packed, s4, scale_2 = nvfp4.quantize(w)
    amax = Fraction(float(np.max(np.abs(w))))
    assert Fraction(float(scale_2)) == Fraction(float(np.float32(float(amax) / 2688.0)))
    sc2 = Fraction(float(scale_2))
    codes = nvfp4.unpack_codes(packed)
    for n in range(3):
        for b in range(2):
            blk = [Fraction(float(v)) for v in w[n, 16 * b:16 * b + 16]]
            bm = max(abs(v) for v in blk)
            s4_ref = _brute_nearest(bm / (6 * sc2), F.E4M3_VALUE_FRAC[:127])
            assert s4[n, b] == s4_ref
            step = F.E4M3_VALUE_FRAC[s4_ref] * sc2
            for j, v in enumerate(blk):
                m = _brute_nearest(abs(v) / step, F.E2M1_MAG_FRAC) if step > 0 else 0
                sgn = 8 if np.signbit(w[n, 16 * b + j]) else 0
                assert codes[n, 16 * b + j] == (sgn | m)


def test_nvfp4_error_bound():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    packed, s4, scale_2 = nvfp4.quantize(w)
    deq = nvfp4.dequantize(packed, s4, scale_2)
    step = np.repeat(F.e4m3_decode(s4), 16, axis=1) * float(scale_2)
    # half the widest e2m1 gap (between 4 and 6) is 1 step; saturation at 6 adds
    # at most 6*(RNE excess of s4), also below 1 step for normal s4
    assert np.all(np.abs(w - deq) <= step + 1e-30)


# ------------------------------------------------------------------ requant
def test_requant_worked_example():
    g = _load("requant_worked_example.json")
    codes = _pack_codes(g["codes"])
    s4 = np.array([[g["s4_code"]]], dtype=np.uint8)
    assert nvfp4.dequantize_units(codes, s4).reshape(-1).tolist() == g["v"]
    codes32 = np.concatenate([codes, codes], axis=1)          # planes need K % 32 == 0
    s4_32 = np.concatenate([s4, s4], axis=1)
    out = requant.requant_2bit(codes32, s4_32)
    assert out["s16"].reshape(-1).tolist() == [g["expect_s16_code"]] * 2
    w2 = requant.dequant_2bit_units(out["sign"], out["mag"], out["s16"]).reshape(-1)[:16]
    assert (w2 / g["expect_s16"]).tolist() == g["expect_q"]
    v = np.array(g["v"], dtype=np.float64)
    assert (v - w2).tolist() == g["expect_delta"]
    assert out["ds4"].reshape(-1).tolist() == [g["expect_ds4_code"]] * 2
    dcodes = nvfp4.unpack_codes(out["dcodes"]).reshape(-1)[:16]
    assert dcodes.tolist() == g["expect_dcodes"]
    assert (F.e2m1_decode(dcodes)).tolist() == g["expect_dcode_values"]


def _random_nvfp4(rng, N, K, zero_frac=0.05):
    codes = rng.integers(0, 16, (N, K), dtype=np.uint8)
    codes[rng.random((N, K)) < zero_frac] = 0
    s4 = rng.integers(0, 127, (N, K // 16), dtype=np.uint8)     # finite, non-negative
    s4[rng.random((N, K // 16)) < 0.05] = 0
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), s4


def test_requant_bruteforce_levels():
    """s16 is the nearest e4m3 to max|v|/3 and q the nearest of {s16, 3 s16} (ties -> 3)."""
    rng = np.random.default_rng(5)
    codes, s4 = _random_nvfp4(rng, 6, 64)
    out = requant.requant_2bit(codes, s4)
    c4 = nvfp4.unpack_codes(codes)
    sign = requant.unpack_bits(out["sign"])
    mag = requant.unpack_bits(out["mag"])
    for n in range(6):
        for b in range(4):
            vals = [F.E2M1_MAG_FRAC[c & 7] * (-1 if c & 8 else 1) * F.E4M3_VALUE_FRAC[s4[n, b]]
                    for c in c4[n, 16 * b:16 * b + 16]]
            bm = max(abs(v) for v in vals)
            s16_ref = _brute_nearest(bm / 3, F.E4M3_VALUE_FRAC[:127])
            assert out["s16"][n, b] == s16_ref
            s = F.E4M3_VALUE_FRAC[s16_ref]
            for j, v in enumerate(vals):
                k = 16 * b + j
                to1, to3 = abs(abs(v) - s), abs(abs(v) - 3 * s)
                assert mag[n, k] == (1 if to3 <= to1 else 0)
                assert sign[n, k] == (c4[n, k] >> 3)


def test_requant_never_zero_and_error_bound():
    rng = np.random.default_rng(6)
    codes, s4 = _random_nvfp4(rng, 32, 128)
    out = requant.requant_2bit(codes, s4)
    s16v = np.repeat(F.e4m3_decode(out["s16"]), 16, axis=1)
    w2 = requant.dequant_2bit_units(out["sign"], out["mag"], out["s16"])
    ok = s16v > 0
    q = w2[ok] / s16v[ok]
    assert set(np.unique(q).tolist()) <= {-3.0, -1.0, 1.0, 3.0}
    v = nvfp4.dequantize_units(codes, s4)
    bmax = np.repeat(np.abs(v).reshape(32, -1, 16).max(axis=2), 16, axis=1)
    unclipped = bmax / 3 <= 448
    assert np.all(np.abs(v - w2)[unclipped] <= s16v[unclipped])


def test_requant_sign_symmetry():
    rng = np.random.default_rng(7)
    codes, s4 = _random_nvfp4(rng, 16, 96)
    neg = codes ^ np.uint8(0x88)                       # flip both nibbles' sign bits
    a = requant.requant_2bit(codes, s4)
    b = requant.requant_2bit(neg, s4)
    assert np.array_equal(b["sign"], ~a["sign"])
    assert np.array_equal(b["mag"], a["mag"])
    assert np.array_equal(b["s16"], a["s16"])
    assert np.array_equal(b["ds4"], a["ds4"])
    ca, cb = nvfp4.unpack_codes(a["dcodes"]), nvfp4.unpack_codes(b["dcodes"])
    nz = (ca & 7) > 0
    assert np.array_equal(cb[nz], ca[nz] ^ 8)
    assert np.all(cb[~nz] == 0) and np.all(ca[~nz] == 0)


def test_delta_reconstruction_bound():
    """W_2bit + deq(delta) reproduces W_nvfp4 to NVFP4 rounding of the residual."""
    rng = np.random.default_rng(8)
    codes, s4 = _random_nvfp4(rng, 32, 128)
    out = requant.requant_2bit(codes, s4)
    v = nvfp4.dequantize_units(codes, s4)
    w2 = requant.dequant_2bit_units(out["sign"], out["mag"], out["s16"])
    dq = nvfp4.dequantize_units(out["dcodes"], out["ds4"])
    d = v - w2
    err = np.abs(d - dq)
    step = np.repeat(F.e4m3_decode(out["ds4"]), 16, axis=1)
    dmax = np.repeat(np.abs(d).reshape(32, -1, 16).max(axis=2), 16, axis=1)
    bound = np.maximum(step, dmax - 6 * step)
    assert np.all(err <= bound)
    normal = step >= 2.0 ** -6
    assert np.all(err[normal] <= step[normal])
    # exact where the residual is itself on the delta grid
    on_grid = np.isin(np.abs(d) / np.where(step > 0, step, 1), F.E2M1_MAG) & (step > 0)
    assert np.all(err[on_grid] == 0)


def test_requant_realistic_weights_roundtrip():
    """NVFP4-quantised N(0, 0.02) weights: the delta restores them almost exactly."""
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, s4, scale_2 = nvfp4.quantize(w)
    out = requant.requant_2bit(codes, s4)
    v = nvfp4.dequantize(codes, s4, scale_2)
    w2 = requant.dequant_2bit(out["sign"], out["mag"], out["s16"], scale_2)
    dq = nvfp4.dequantize(out["dcodes"], out["ds4"], scale_2)
    rel2 = np.linalg.norm(v - w2) / np.linalg.norm(v)
    relf = np.linalg.norm(v - w2 - dq) / np.linalg.norm(v)
    assert 0.2 < rel2 < 0.6          # 2-bit alone is coarse
    assert relf < 0.1 * rel2         # the FP4 residual recovers >90% of it


# ---------------------------------------------------------------- FP8 block-quant input
def _random_fp8(rng, N, K, nbs_scale=1.0):
    codes = rng.integers(0, 256, (N, K), dtype=np.uint8)
    nan = (codes & 0x7F) == 0x7F
    codes[nan] ^= 1                                       # the NaN codes are not weights
    codes[0, :5] = [0x00, 0x80, 0x7E, 0xFE, 0x01]          # +0, -0, +-448, smallest subnormal
    bs = (rng.random(((N + 127) // 128, (K + 127) // 128)) * 0.02 + 0.001).astype(np.float32) * np.float32(nbs_scale)
    return codes, bs


def _fp8_wide_scales(rng):
    """Three rows of 384 codes under three block scales each, the scales spread over 2^-120 ..
    2^20 with one fp32 subnormal and one zero: blocks far below the matrix's largest (s16 = 0 or
    a subnormal s16) next to the top block."""
    codes, _ = _random_fp8(rng, 3, 384)
    codes[2, 256:272] = codes[2, 256]                        # sixteen equal codes
    bs = np.array([[np.ldexp(1.37, 20), np.ldexp(1.9, -7), np.float32(3e-43)]], np.float32)
    bs2 = np.array([[np.ldexp(1.1, -120), 0.0, np.ldexp(1.61, 13)]], np.float32)
    return codes, bs, bs2


@pytest.mark.parametrize("case", ["narrow", "wide_a", "wide_b"])
def test_fp8_requant_matches_exact_fractions(case):
    """Every integer output of the fp64 FP8 requant against the same rule evaluated in exact
    rational arithmetic (Fraction), weight by weight; block scales of one magnitude, then spread
    over 140 binades (the exactness of the fp64 residual and every fp64 comparison is claimed for
    any scales, so it is pinned there too)."""
    rng = np.random.default_rng(21)
    if case == "narrow":
        codes, bs = _random_fp8(rng, 3, 64)
        bs[:] = rng.choice(np.array([0.0078125, 0.3, 1.7e-3], np.float32), size=bs.shape)
    else:
        codes, bs_a, bs_b = _fp8_wide_scales(rng)
        bs = bs_a if case == "wide_a" else bs_b
    out = requant.requant_fp8_2bit(codes, bs)
    s2 = Fraction(float(out["scale_2"]))
    N, K = codes.shape
    sign = requant.unpack_bits(out["sign"]); mag = requant.unpack_bits(out["mag"])
    dc = np.zeros((N, K), np.uint8)
    dc[:, 0::2] = out["dcodes"] & 15; dc[:, 1::2] = out["dcodes"] >> 4
    for n in range(N):
        wf = [F.E4M3_VALUE_FRAC[int(c) & 0x7F] * Fraction(float(bs[n // 128, k // 128])) * (-1 if c & 0x80 else 1)
              for k, c in enumerate(codes[n])]
        for b in range(K // 16):
            blk = wf[16 * b:16 * b + 16]
            s16 = F.e4m3_rne_fraction(max(abs(x) for x in blk) / (3 * s2))
            assert out["s16"][n, b] == s16
            lvl = F.E4M3_VALUE_FRAC[s16] * s2
            d = []
            for j, x in enumerate(blk):
                k = 16 * b + j
                assert sign[n, k] == (codes[n, k] >> 7)
                m = abs(x) >= 2 * lvl
                assert mag[n, k] == m
                q = (3 if m else 1) * lvl * (-1 if sign[n, k] else 1)
                d.append(x - q)
            dmax = max(abs(x) for x in d)
            ds4 = F.e4m3_rne_fraction(dmax / (6 * s2)) if dmax else 0
            assert out["ds4"][n, b] == ds4
            step = F.E4M3_VALUE_FRAC[ds4] * s2
            for j, x in enumerate(d):
                mg = F.e2m1_rne_fraction(abs(x) / step) if step else 0
                code = mg | (8 if (x < 0 and mg) else 0)
                assert dc[n, 16 * b + j] == code


def test_fp8_requant_scale_and_sign_invariance():
    """Doubling every block scale doubles scale_2 exactly and changes no plane, scale or delta
    code; negating every weight flips the sign plane and the delta signs only."""
    rng = np.random.default_rng(22)
    codes, bs = _random_fp8(rng, 200, 96)
    a = requant.requant_fp8_2bit(codes, bs)
    b = requant.requant_fp8_2bit(codes, bs * np.float32(2))
    assert np.float32(b["scale_2"]) == np.float32(2) * np.float32(a["scale_2"])
    for key in ("sign", "mag", "s16", "dcodes", "ds4"):
        assert np.array_equal(a[key], b[key]), key
    c = requant.requant_fp8_2bit(codes ^ np.uint8(0x80), bs)
    assert np.array_equal(c["sign"], ~a["sign"]) and np.array_equal(c["mag"], a["mag"])
    assert np.array_equal(c["s16"], a["s16"]) and np.array_equal(c["ds4"], a["ds4"])
    flip = np.zeros_like(a["dcodes"])
    lo, hi = a["dcodes"] & 15, a["dcodes"] >> 4
    flip |= np.where((lo & 7) != 0, 8, 0).astype(np.uint8)
    flip |= np.where((hi & 7) != 0, 0x80, 0).astype(np.uint8)
    assert np.array_equal(c["dcodes"], a["dcodes"] ^ flip)


def test_fp8_requant_top_block_and_zero_matrix():
    rng = np.random.default_rng(23)
    codes, bs = _random_fp8(rng, 4, 64)
    out = requant.requant_fp8_2bit(codes, bs)
    w = requant.fp8_dequantize(codes, bs)
    top = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert out["s16"][top[0], top[1] // 16] == 126                  # the largest block: s16 = 448
    z = requant.requant_fp8_2bit(np.zeros((2, 32), np.uint8), np.ones((1, 1), np.float32))
    assert z["scale_2"] == 0 and not z["s16"].any() and not z["ds4"].any() and not z["dcodes"].any()
    assert (z["mag"] == 0xFFFFFFFF).all()                             # |q| = 3 on a zero scale


# ---------------------------------------------------------------- MXFP4 (FP4 experts) input
def _random_mxfp4(rng, N, K, lo=110, hi=140):
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    codes[0, :2] = [0x80, 0x7F]                            # (+0, -0), (-6, +6)
    e8m0 = rng.integers(lo, hi, (N, K // 32)).astype(np.uint8)
    return codes, e8m0


def test_mxfp4_requant_matches_exact_fractions():
    """Every integer output of the fp64 MXFP4 requant against the same rule on weights decoded
    in exact rational arithmetic (Fraction) from the codes and E8M0 exponents, weight by weight;
    exponents span the whole E8M0 range except NaN."""
    rng = np.random.default_rng(31)
    codes, e8m0 = _random_mxfp4(rng, 3, 64)
    e8m0[0] = [0, 254]                                     # 2^-127 and 2^127
    e8m0[1] = [127, 126]
    e8m0[2] = [1, 3]
    for rows in ([0], [1, 2]):
        c, e = codes[rows], e8m0[rows]
        out = requant.requant_mxfp4_2bit(c, e)
        N, K = c.shape[0], c.shape[1] * 2
        nib = np.zeros((N, K), np.uint8)
        nib[:, 0::2] = c & 15; nib[:, 1::2] = c >> 4
        wf = [[F.E2M1_MAG_FRAC[int(x) & 7] * Fraction(2) ** (int(e[n, k // 32]) - 127) * (-1 if x & 8 else 1)
               for k, x in enumerate(nib[n])] for n in range(N)]
        amax = max(abs(x) for r in wf for x in r)
        assert Fraction(float(out["scale_2"])) == Fraction(float(np.float32(float(amax / 1344))))
        s2 = Fraction(float(out["scale_2"]))
        sign = requant.unpack_bits(out["sign"]); mag = requant.unpack_bits(out["mag"])
        dc = np.zeros((N, K), np.uint8)
        dc[:, 0::2] = out["dcodes"] & 15; dc[:, 1::2] = out["dcodes"] >> 4
        for n in range(N):
            for b in range(K // 16):
                blk = wf[n][16 * b:16 * b + 16]
                bm = max(abs(x) for x in blk)
                s16 = F.e4m3_rne_fraction(bm / (3 * s2)) if bm else 0
                assert out["s16"][n, b] == s16
                lvl = F.E4M3_VALUE_FRAC[s16] * s2
                d = []
                for j, x in enumerate(blk):
                    k = 16 * b + j
                    assert sign[n, k] == (nib[n, k] >> 3)
                    m = abs(x) >= 2 * lvl
                    assert mag[n, k] == m
                    d.append(x - (3 if m else 1) * lvl * (-1 if sign[n, k] else 1))
                dmax = max(abs(x) for x in d)
                ds4 = F.e4m3_rne_fraction(dmax / (6 * s2)) if dmax else 0
                assert out["ds4"][n, b] == ds4
                step = F.E4M3_VALUE_FRAC[ds4] * s2
                for j, x in enumerate(d):
                    mg = F.e2m1_rne_fraction(abs(x) / step) if step else 0
                    assert dc[n, 16 * b + j] == (mg | (8 if (x < 0 and mg) else 0))


def test_mxfp4_requant_equals_fp8_on_the_same_weights():
    """An MXFP4 matrix whose weights are all e4m3 values (exponents 2^-6 .. 2^6) and the FP8
    block-quant matrix holding the same weights (block scale 1) give the same scale_2, planes,
    s16 and delta: both inputs go through one rule on the exact weights."""
    rng = np.random.default_rng(32)
    N, K = 130, 96
    codes, e8m0 = _random_mxfp4(rng, N, K, lo=121, hi=134)
    w = requant.mxfp4_dequantize(codes, e8m0)
    e4 = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    lut = {}
    for c in range(256):
        if (c & 0x7F) != 0x7F:
            lut.setdefault((float(abs(e4[c])), c >> 7), c)
    nib = np.zeros((N, K), np.uint8)
    nib[:, 0::2] = codes & 15; nib[:, 1::2] = codes >> 4
    f8 = np.array([[lut[(float(abs(w[n, k])), int(nib[n, k] >> 3))] for k in range(K)] for n in range(N)], np.uint8)
    a = requant.requant_mxfp4_2bit(codes, e8m0)
    b = requant.requant_fp8_2bit(f8, np.ones((2, 1), np.float32))
    assert a["scale_2"] == b["scale_2"]
    for key in ("sign", "mag", "s16", "dcodes", "ds4"):
        assert np.array_equal(a[key], b[key]), key


def test_mxfp4_requant_scale_and_sign_invariance():
    """Adding 1 to every exponent doubles scale_2 exactly and changes nothing else; flipping
    every code's sign bit flips the sign plane and the delta signs only."""
    rng = np.random.default_rng(33)
    codes, e8m0 = _random_mxfp4(rng, 200, 96)
    a = requant.requant_mxfp4_2bit(codes, e8m0)
    b = requant.requant_mxfp4_2bit(codes, e8m0 + np.uint8(1))
    assert np.float32(b["scale_2"]) == np.float32(2) * np.float32(a["scale_2"])
    for key in ("sign", "mag", "s16", "dcodes", "ds4"):
        assert np.array_equal(a[key], b[key]), key
    c = requant.requant_mxfp4_2bit(codes ^ np.uint8(0x88), e8m0)
    assert np.array_equal(c["sign"], ~a["sign"]) and np.array_equal(c["mag"], a["mag"])
    assert np.array_equal(c["s16"], a["s16"]) and np.array_equal(c["ds4"], a["ds4"])
    lo, hi = a["dcodes"] & 15, a["dcodes"] >> 4
    flip = np.where((lo & 7) != 0, 8, 0).astype(np.uint8) | np.where((hi & 7) != 0, 0x80, 0).astype(np.uint8)
    assert np.array_equal(c["dcodes"], a["dcodes"] ^ flip)


def test_mxfp4_requant_top_block_and_zero_matrix():
    rng = np.random.default_rng(34)
    codes, e8m0 = _random_mxfp4(rng, 4, 64)
    out = requant.requant_mxfp4_2bit(codes, e8m0)
    w = requant.mxfp4_dequantize(codes, e8m0)
    top = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert out["s16"][top[0], top[1] // 16] == 126                  # the largest block: s16 = 448
    z = requant.requant_mxfp4_2bit(np.zeros((2, 16), np.uint8), np.full((2, 1), 127, np.uint8))
    assert z["scale_2"] == 0 and not z["s16"].any() and not z["ds4"].any() and not z["dcodes"].any()
    assert (z["mag"] == 0xFFFFFFFF).all()
