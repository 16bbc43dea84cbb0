"""fp32 -> NVFP4 quantiser: the input format of the expert weights.

README "Frontier MoE on consumer Blackwell (SM120)", §"GLM-5.2 (753B)" ¶1:
modelopt NVFP4 experts are e2m1 values x an e4m3 scale per block of 16 along
K x one fp32 per-tensor scale_2.  The pages give no formula beyond that; this
is the plainest modelopt-style reading, used only to make inputs:

  amax    = max |W| over the tensor
  scale_2 = fp32(amax / 2688)              2688 = 6 (e2m1 max) * 448 (e4m3 max)
  s4[b]   = e4m3 satfinite RNE( max_{k in b} |w_k| / (6 * scale_2) )
  code_k  = sign(w_k) | e2m1 satfinite RNE( |w_k| / (s4[b] * scale_2) )

Ties go to the even code, the sign is the sign bit of w (so -0 stays -0), a
block whose s4 is 0 (or a tensor whose amax is 0) gets codes +-0.  Byte
packing: the low nibble holds the even k.
"""
from __future__ import annotations

import numpy as np

from .formats import E4M3_POS, e2m1_rne_ratio, e4m3_rne_ratio


def quantize(w: np.ndarray):
    """One [N, K] fp32 matrix -> (codes u8 [N, K/2], s4 u8 [N, K/16], scale_2 fp32)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 16 == 0
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    scale_2 = np.float32(amax) / np.float32(2688.0)          # one fp32 rounding
    a = np.abs(w).astype(np.float64)
    bmax = a.reshape(N, K // 16, 16).max(axis=2)
    if scale_2 > 0:
        s4 = e4m3_rne_ratio(bmax, 6.0 * np.float64(scale_2))
    else:
        s4 = np.zeros((N, K // 16), dtype=np.uint8)
    s4v = E4M3_POS[s4.astype(np.int64)]                      # exact, >= 0
    step = np.repeat(s4v, 16, axis=1) * np.float64(scale_2)  # exact product
    mag = np.zeros((N, K), dtype=np.uint8)
    nz = step > 0
    mag[nz] = e2m1_rne_ratio(a[nz], step[nz])
    sign = np.signbit(w).astype(np.uint8)
    code = (sign << 3) | mag
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, s4.astype(np.uint8), np.float32(scale_2)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes (low nibble first)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 15
    out[..., 1::2] = packed >> 4
    return out


def dequantize_units(packed: np.ndarray, s4: np.ndarray) -> np.ndarray:
    """NVFP4 values in units of scale_2 (fp64, exact): e2m1(code) * e4m3(s4)."""
    from .formats import e2m1_decode, e4m3_decode
    codes = unpack_codes(packed)
    return e2m1_decode(codes) * np.repeat(e4m3_decode(s4), 16, axis=-1)


def dequantize(packed: np.ndarray, s4: np.ndarray, scale_2) -> np.ndarray:
    return dequantize_units(packed, s4) * np.float64(scale_2)
