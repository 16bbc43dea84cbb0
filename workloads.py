"""Seeded synthetic inputs for the 2-bit MoE expert layer.

This module draws random numbers and nothing else: router logits, bf16
activations, fp32 expert weights, the delta-cache expert set and the per-token
gate mask.  It holds none of the method's arithmetic (no quantisation, no
routing, no GEMM), so both the CPU oracle and the CUDA path can take their
inputs from here without sharing any of the computation they are checked on.

Workloads (shapes and value recipes of the MoE layers described by the
vLLM-Moet README, "Frontier MoE on consumer Blackwell (SM120)", §GLM-5.2,
§DeepSeek-V4-Flash, §Kimi-K2.7-Code, and of a tiny correctness layer):

  tiny        T=4, H=256, I=128, E=8, k=2; W ~ N(0, 0.02); delta set {0, 3};
              gate = token 1 only.
  dsv3_decode H=7168, I=2048, E=256, k=8, T in {1, 8, 64}; W ~ N(0, 0.02);
              32 delta experts drawn uniformly; gate ~ Bernoulli(0.1).
  dsv3_prefill  as dsv3_decode with T=4096 and a Zipf(s=1.1) logit bias
              over a random permutation of the experts.
  glm_decode  H=6144, I=2048, E=256, k=8, T=8; W ~ Student-t(nu=4) scaled
              to std 0.02; 64 delta experts; every token gated.
  kimi_layer  H=7168, I=2048, E=384, k=8, T=256; uniform routing;
              W ~ Student-t(nu=4) at std 0.02; no delta table.

Draw order from the main stream ``numpy.random.default_rng(seed)``:
logits noise, Zipf permutation (prefill only), activations, delta set, gate.
Weights come from an independent stream per (expert, FC) so that any one
expert can be regenerated alone: ``default_rng([seed, 1000 + e, fc])``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["LayerConfig", "CONFIGS", "draw_logits", "draw_x_bf16", "draw_weight",
           "draw_delta_set", "draw_gate", "bf16_bits_to_f32", "f32_to_bf16_bits",
           "draw_plane_matrix", "draw_plane_scale2", "draw_delta_matrix"]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    dist: str            # "normal" or "student_t4"
    n_delta: int         # experts held in the delta cache
    gate: str            # "token1", "bernoulli0.1", "all", "none"
    zipf: float = 0.0    # Zipf exponent of the logit bias (0 = none)
    seed: int = 0


CONFIGS = {
    "tiny": LayerConfig("tiny", 4, 256, 128, 8, 2, "normal", 2, "token1"),
    "dsv3_decode_t1": LayerConfig("dsv3_decode_t1", 1, 7168, 2048, 256, 8, "normal", 32, "bernoulli0.1"),
    "dsv3_decode_t8": LayerConfig("dsv3_decode_t8", 8, 7168, 2048, 256, 8, "normal", 32, "bernoulli0.1"),
    "dsv3_decode_t64": LayerConfig("dsv3_decode_t64", 64, 7168, 2048, 256, 8, "normal", 32, "bernoulli0.1"),
    "dsv3_prefill": LayerConfig("dsv3_prefill", 4096, 7168, 2048, 256, 8, "normal", 32, "bernoulli0.1", zipf=1.1),
    "glm_decode": LayerConfig("glm_decode", 8, 6144, 2048, 256, 8, "student_t4", 64, "all"),
    "kimi_layer": LayerConfig("kimi_layer", 256, 7168, 2048, 384, 8, "student_t4", 0, "none"),
}


def main_rng(cfg: LayerConfig) -> np.random.Generator:
    return np.random.default_rng(cfg.seed)


def draw_logits(rng: np.random.Generator, cfg: LayerConfig) -> np.ndarray:
    """Router logits [T, E] fp32: N(0, 1), plus log p_rank(e) for the Zipf case.

    The Zipf bias is b_e = ln p_r with p_r proportional to r**-s over ranks
    r = 1..E, and rank(e) a random permutation, so that a softmax of the bias
    alone is the Zipf pmf.
    """
    logits = rng.standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if cfg.zipf > 0.0:
        ranks = rng.permutation(cfg.E) + 1
        p = ranks.astype(np.float64) ** (-cfg.zipf)
        p /= p.sum()
        logits = (logits + np.log(p).astype(np.float32)[None, :]).astype(np.float32)
    return logits


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def draw_x_bf16(rng: np.random.Generator, cfg: LayerConfig) -> np.ndarray:
    """Activations [T, H] as bf16 bit patterns (uint16), N(0, 1) before rounding."""
    x = rng.standard_normal((cfg.T, cfg.H), dtype=np.float32)
    return f32_to_bf16_bits(x)


def weight_rng(cfg: LayerConfig, expert: int, fc: int) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, 1000 + expert, fc])


def draw_weight(cfg: LayerConfig, expert: int, fc: int) -> np.ndarray:
    """fp32 weight of one expert: fc=1 -> [2I, H] (gate rows then up rows), fc=2 -> [H, I]."""
    shape = (2 * cfg.I, cfg.H) if fc == 1 else (cfg.H, cfg.I)
    rng = weight_rng(cfg, expert, fc)
    if cfg.dist == "normal":
        w = rng.standard_normal(shape, dtype=np.float32) * np.float32(0.02)
    elif cfg.dist == "student_t4":
        w = (rng.standard_t(4.0, size=shape) * (0.02 / math.sqrt(2.0))).astype(np.float32)
    else:
        raise ValueError(cfg.dist)
    return w.astype(np.float32)


def draw_delta_set(rng: np.random.Generator, cfg: LayerConfig) -> np.ndarray:
    """Sorted expert ids held in the delta cache."""
    if cfg.name == "tiny":
        return np.array([0, 3], dtype=np.int32)
    if cfg.n_delta == 0:
        return np.zeros(0, dtype=np.int32)
    return np.sort(rng.choice(cfg.E, size=cfg.n_delta, replace=False)).astype(np.int32)


def draw_gate(rng: np.random.Generator, cfg: LayerConfig) -> np.ndarray:
    """Per-token gate mask [T] uint8 (1 = token runs with the FP4 delta)."""
    if cfg.gate == "token1":
        g = np.zeros(cfg.T, dtype=np.uint8)
        g[1] = 1
        return g
    if cfg.gate == "bernoulli0.1":
        return (rng.random(cfg.T) < 0.1).astype(np.uint8)
    if cfg.gate == "all":
        return np.ones(cfg.T, dtype=np.uint8)
    return np.zeros(cfg.T, dtype=np.uint8)


def draw_layer_inputs(cfg: LayerConfig):
    """Logits, x (bf16 bits), delta set and gate, in the documented draw order."""
    rng = main_rng(cfg)
    logits = draw_logits(rng, cfg)
    x = draw_x_bf16(rng, cfg)
    dset = draw_delta_set(rng, cfg)
    gate = draw_gate(rng, cfg)
    return logits, x, dset, gate


def delta_slot_table(E: int, dset: np.ndarray) -> np.ndarray:
    """expert -> slot in the delta pool (-1 = not cached); slots follow dset order."""
    slot = np.full(E, -1, dtype=np.int32)
    slot[dset] = np.arange(len(dset), dtype=np.int32)
    return slot


# ---------------------------------------------------------------- random plane sets
# Any sign and magnitude bits with any e4m3 block scales form a valid 2-bit
# expert matrix, so the full-size parity checks draw the planes directly (the
# oracle's own requantisation of 17 G weights would take hours on a CPU).  Each
# part of each (expert, FC) matrix has its own stream, so any one part can be
# regenerated alone: default_rng([seed, 2000 + e, fc, part]).

def draw_plane_matrix(seed: int, expert: int, fc: int, N: int, K: int, heavy: bool = False):
    """(sign [N, K/32] u32, mag [N, K/32] u32, s16 [N, K/16] u8) of one expert matrix.

    Bits are uniform.  Block-scale codes (e4m3fn) are a mixture over the whole
    finite range: 90 % in the upper band a requantised layer mostly holds
    (codes 96..126, i.e. 32..448; with ``heavy`` 72..126, i.e. 4..448, a
    Student-t-like spread of block maxima), 5 % small normal codes below that
    band, 4 % subnormal codes 1..7 and 1 % zero blocks."""
    def g(part):
        return np.random.default_rng([seed, 2000 + expert, fc, part])
    sign = g(0).integers(0, 2 ** 32, (N, K // 32), dtype=np.uint32)
    mag = g(1).integers(0, 2 ** 32, (N, K // 32), dtype=np.uint32)
    r = g(2)
    nb = (N, K // 16)
    lo = 72 if heavy else 96
    s16 = r.integers(lo, 127, nb, dtype=np.uint8)
    u = r.random(nb)
    small = r.integers(8, lo, nb, dtype=np.uint8)
    sub = r.integers(1, 8, nb, dtype=np.uint8)
    s16 = np.where(u < 0.05, small, s16)
    s16 = np.where((u >= 0.05) & (u < 0.09), sub, s16)
    s16 = np.where((u >= 0.09) & (u < 0.10), np.uint8(0), s16).astype(np.uint8)
    return sign, mag, s16


def draw_plane_scale2(seed: int, fc: int, E: int, K: int) -> np.ndarray:
    """Per-expert fp32 scale_2 [E] for draw_plane_matrix planes: uniform in
    [0.5, 1.5] / (450 sqrt(K)) (450 is about the rms of q s16 for the upper band),
    so that a unit-variance activation row gives O(1) outputs."""
    r = np.random.default_rng([seed, 3000, fc])
    return (r.uniform(0.5, 1.5, E) / (450.0 * math.sqrt(K))).astype(np.float32)


def draw_delta_matrix(seed: int, slot: int, fc: int, N: int, K: int):
    """(codes [N, K/2] u8, s4 [N, K/16] u8) of one delta-pool slot: uniform code
    bytes; scale codes 64..110 (0.125..224, the range of a residual's block
    maxima over 6) with 2 % zero blocks."""
    r = np.random.default_rng([seed, 4000 + slot, fc])
    codes = r.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s4 = r.integers(64, 111, (N, K // 16), dtype=np.uint8)
    s4[r.random(s4.shape) < 0.02] = 0
    return codes, s4
