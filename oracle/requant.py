"""Load-time requantisation NVFP4 -> sign-symmetric 2-bit planes, and the NVFP4 delta.

README "Frontier MoE on consumer Blackwell (SM120)", §"GLM-5.2 (753B)" ¶1 and
§"How it fits -- 2-bit experts at FP4 quality" (bullets 1-2, last ¶): the
loader dequantises modelopt NVFP4 experts exactly and requantises them to a
sign-symmetric 2-bit codebook; an FP4 "delta" restores NVFP4 precision for
experts held in the delta cache.  The pages print the levels {-4,-1,1,4};
this library fixes the codebook q in {-3,-1,+1,+3} (no zero level).

Everything is in units of the tensor's scale_2, where an NVFP4 weight is the
exact number v = e2m1(code) * e4m3(s4).  Per block b of 16 along K:

  s16[b]  = e4m3 satfinite RNE( max_{k in b} |v_k| / 3 )
  sign_k  = sign bit of the NVFP4 code (so -0 maps to the negative side)
  mag_k   = |v_k| >= 2 * s16[b]        (|q| = 3; the tie goes to 3)
  W2_k    = (sign ? -1 : +1) * (mag ? 3 : 1) * s16[b]          (x scale_2)

Delta (the residual on the same scale_2):

  d_k     = v_k - W2_k                                     (exact in fp64)
  s4d[b]  = e4m3 satfinite RNE( max_{k in b} |d_k| / 6 )
  dcode_k = sign(d_k) | e2m1 satfinite RNE(|d_k| / s4d[b]);  a zero
            magnitude is written as +0, and s4d = 0 gives all +0.

Plane layout: row-major [N, K/32] uint32, bit j of word w holds weight
k = 32 w + j (least significant bit first); sign bit 1 = negative, mag bit 1 =
|q| = 3.  Delta codes pack two per byte, low nibble = even k.
"""
from __future__ import annotations

import numpy as np

from .formats import E4M3_POS, e2m1_decode, e2m1_rne_ratio, e4m3_rne_ratio, e4m3_decode
from .nvfp4 import dequantize_units, unpack_codes


def pack_bits(bits: np.ndarray) -> np.ndarray:
    """[N, K] of 0/1 -> [N, K/32] uint32, bit j of word w = element 32w + j."""
    bits = np.asarray(bits, dtype=np.uint64)
    N, K = bits.shape
    assert K % 32 == 0
    b = bits.reshape(N, K // 32, 32)
    weights = np.uint64(1) << np.arange(32, dtype=np.uint64)
    return (b * weights).sum(axis=2).astype(np.uint32)


def unpack_bits(words: np.ndarray) -> np.ndarray:
    """[N, K/32] uint32 -> [N, K] uint8 of 0/1."""
    words = np.asarray(words, dtype=np.uint32)
    shifts = np.arange(32, dtype=np.uint32)
    b = (words[..., None] >> shifts) & np.uint32(1)
    return b.reshape(words.shape[:-1] + (words.shape[-1] * 32,)).astype(np.uint8)


def requant_2bit(codes: np.ndarray, s4: np.ndarray, want_delta: bool = True):
    """One [N, K] NVFP4 matrix (codes [N, K/2], s4 [N, K/16]) -> planes (+ delta).

    Returns dict(sign [N,K/32] u32, mag [N,K/32] u32, s16 [N,K/16] u8) and, if
    ``want_delta``, also dcodes [N, K/2] u8 and ds4 [N, K/16] u8.
    """
    v = dequantize_units(codes, s4)                    # exact fp64, units of scale_2
    N, K = v.shape
    av = np.abs(v)
    bmax = av.reshape(N, K // 16, 16).max(axis=2)
    s16 = e4m3_rne_ratio(bmax, 3.0)
    s16v = np.repeat(E4M3_POS[s16.astype(np.int64)], 16, axis=1)
    sign = (unpack_codes(codes) >> 3).astype(np.uint8)
    mag = (av >= 2.0 * s16v).astype(np.uint8)
    out = dict(sign=pack_bits(sign), mag=pack_bits(mag), s16=s16.astype(np.uint8))
    if want_delta:
        w2 = np.where(sign == 1, -1.0, 1.0) * np.where(mag == 1, 3.0, 1.0) * s16v
        d = v - w2                                      # exact: both are short dyadics
        ad = np.abs(d)
        dmax = ad.reshape(N, K // 16, 16).max(axis=2)
        ds4 = e4m3_rne_ratio(dmax, 6.0)
        step = np.repeat(E4M3_POS[ds4.astype(np.int64)], 16, axis=1)
        dmag = np.zeros((N, K), dtype=np.uint8)
        nz = step > 0
        dmag[nz] = e2m1_rne_ratio(ad[nz], step[nz])
        dsign = ((d < 0) & (dmag > 0)).astype(np.uint8)
        dcode = (dsign << 3) | dmag
        out["dcodes"] = (dcode[:, 0::2] | (dcode[:, 1::2] << 4)).astype(np.uint8)
        out["ds4"] = ds4.astype(np.uint8)
    return out


def dequant_2bit_units(sign: np.ndarray, mag: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """2-bit planes -> fp64 weights in units of scale_2."""
    sb = unpack_bits(sign)
    mb = unpack_bits(mag)
    q = np.where(sb == 1, -1.0, 1.0) * np.where(mb == 1, 3.0, 1.0)
    return q * np.repeat(e4m3_decode(s16), 16, axis=-1)


def dequant_2bit(sign, mag, s16, scale_2) -> np.ndarray:
    return dequant_2bit_units(sign, mag, s16) * np.float64(scale_2)


# ---------------------------------------------------------------- FP8 block-quant input
FP8_BLOCK = 128          # DeepSeek-style block quantisation: one fp32 scale per 128 x 128 block
S16_TOP = 3 * 448        # scale_2 = amax / 1344: the largest block's s16 lands at 448


def fp8_dequantize(codes: np.ndarray, bscale: np.ndarray) -> np.ndarray:
    """[N, K] e4m3 codes with fp32 block scales [ceil(N/128), ceil(K/128)] -> exact fp64 weights
    (an e4m3 value has 4 significant bits, an fp32 scale 24: the product is exact in fp64)."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, K = codes.shape
    bs = np.asarray(bscale, dtype=np.float32).astype(np.float64)
    rep = np.repeat(np.repeat(bs, FP8_BLOCK, axis=0)[:N], FP8_BLOCK, axis=1)[:, :K]
    return e4m3_decode(codes) * rep


def fp8_scale_2(codes: np.ndarray, bscale: np.ndarray) -> np.float32:
    """Per-matrix scale_2 for an FP8 block-quant matrix: fp32(fp64(amax) / 1344), i.e. the fp64
    quotient rounded to nearest, then to the nearest fp32 (the two roundings define it)."""
    amax = float(np.abs(fp8_dequantize(codes, bscale)).max())
    return np.float32(np.float64(amax) / np.float64(S16_TOP))


def requant_fp8_2bit(codes: np.ndarray, bscale: np.ndarray, want_delta: bool = True):
    """One [N, K] FP8 block-quant matrix -> scale_2, 2-bit planes (+ NVFP4 delta).
    The e4m3 NaN codes (0x7F, 0xFF) are not valid weights.

    README "Frontier MoE on consumer Blackwell (SM120)", §"How it fits -- 2-bit experts at FP4
    quality", last paragraph: FP8 block-quant checkpoints are requantised to the sign-symmetric
    codebook at load, as the NVFP4 ones are.  The pages give no formula for this input; the
    reading here is the NVFP4 rule applied to the exact FP8 weights W with a per-matrix
    scale_2 = amax / (3 * 448) (see fp8_scale_2 and requant_exact_2bit).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    return requant_exact_2bit(fp8_dequantize(codes, bscale), (codes >> 7).astype(np.uint8), want_delta)


def requant_exact_2bit(w: np.ndarray, sign: np.ndarray, want_delta: bool = True):
    """The NVFP4 rule applied to exact weights W [N, K] (fp64) with their sign bits [N, K]:

      scale_2 = fp32( fp64(max |W|) / 1344 )                 (the largest block's s16 is 448)
      s16[b]  = e4m3 satfinite RNE( max_b |W| / (3 scale_2) )
      sign_k  = the input's sign bit (so -0 maps to the negative side)
      mag_k   = |W_k| >= 2 s16[b] scale_2
      d_k     = W_k - q_k s16[b] scale_2                    (exact in fp64)
      ds4[b]  = e4m3 satfinite RNE( max_b |d| / (6 scale_2) )
      dcode_k = sign(d_k) | e2m1 satfinite RNE( |d_k| / (ds4[b] scale_2) ), zero as +0.

    Every ratio is rounded once by exact comparison (formats._rne_ratio): all products of
    the short significands involved are exact in fp64.  A zero block (or matrix) gets s16 = 0.
    """
    w = np.asarray(w, dtype=np.float64)
    sign = np.asarray(sign, dtype=np.uint8)
    N, K = w.shape
    assert K % 32 == 0
    aw = np.abs(w)
    sc2 = np.float32(np.float64(aw.max()) / np.float64(S16_TOP))
    s2 = np.float64(sc2)
    bmax = aw.reshape(N, K // 16, 16).max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        s16 = np.where(bmax > 0, e4m3_rne_ratio(bmax, 3.0 * s2), 0)   # a zero block (or matrix): 0
    lvl = np.repeat(E4M3_POS[s16.astype(np.int64)], 16, axis=1) * s2      # s16 scale_2, exact
    mag = (aw >= 2.0 * lvl).astype(np.uint8)
    out = dict(scale_2=sc2, sign=pack_bits(sign), mag=pack_bits(mag), s16=s16.astype(np.uint8))
    if want_delta:
        w2 = np.where(sign == 1, -1.0, 1.0) * np.where(mag == 1, 3.0, 1.0) * lvl
        d = w - w2
        ad = np.abs(d)
        dmax = ad.reshape(N, K // 16, 16).max(axis=2)
        with np.errstate(divide="ignore", invalid="ignore"):
            ds4 = np.where(dmax > 0, e4m3_rne_ratio(dmax, 6.0 * s2), 0)
        step = np.repeat(E4M3_POS[ds4.astype(np.int64)], 16, axis=1) * s2
        dmag = np.zeros((N, K), dtype=np.uint8)
        nz = step > 0
        dmag[nz] = e2m1_rne_ratio(ad[nz], step[nz])
        dsign = ((d < 0) & (dmag > 0)).astype(np.uint8)
        dcode = (dsign << 3) | dmag
        out["dcodes"] = (dcode[:, 0::2] | (dcode[:, 1::2] << 4)).astype(np.uint8)
        out["ds4"] = ds4.astype(np.uint8)
    return out


# ---------------------------------------------------------------- MXFP4 (FP4 experts) input
MX_BLOCK = 32            # OCP microscaling: one E8M0 scale per 32 consecutive weights along K
E8M0_BIAS = 127


def mxfp4_dequantize(codes: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """[N, K/2] e2m1 codes (low nibble = even k) with E8M0 scales [N, K/32] -> exact fp64
    weights W = e2m1(code) * 2^(e - 127).  The E8M0 NaN code 0xFF is not a valid scale."""
    e8m0 = np.asarray(e8m0, dtype=np.uint8)
    assert not (e8m0 == 0xFF).any(), "E8M0 0xFF (NaN) is not a weight scale"
    v = e2m1_decode(unpack_codes(codes))
    return v * np.repeat(np.ldexp(1.0, e8m0.astype(np.int64) - E8M0_BIAS), MX_BLOCK, axis=1)


def requant_mxfp4_2bit(codes: np.ndarray, e8m0: np.ndarray, want_delta: bool = True):
    """One [N, K] MXFP4 matrix -> scale_2, 2-bit planes (+ NVFP4 delta).

    README "Frontier MoE on consumer Blackwell (SM120)", §"How it fits -- 2-bit experts at FP4
    quality", last paragraph: checkpoints with FP4 experts (DeepSeek-V4-Flash) load by a code
    remap.  The pages name no format and no formula.  Readings: the FP4 experts are OCP MXFP4
    (an e2m1 code per weight, one power-of-two E8M0 scale per 32 weights along K), and the remap
    is the same rule as the FP8 input -- the NVFP4 rule on the exact weights with
    scale_2 = amax / 1344 (requant_exact_2bit).  The sign plane is the e2m1 sign bit; the
    magnitude plane depends only on each code, its block's largest code and exponent, and
    scale_2: it is a remap of the codes.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    sign = (unpack_codes(codes) >> 3).astype(np.uint8)
    return requant_exact_2bit(mxfp4_dequantize(codes, e8m0), sign, want_delta)
