"""The oracle's layer forward over one shard of the experts, for a spawn process pool.

The full-size parity checks compare sampled tokens of the DeepSeek-V3, GLM and
1T-class layers with the fp64 oracle.  Dequantising one expert of those layers
in fp64 takes about a second, and a sample of 8 tokens routes to up to 64
experts, so the experts are split over worker processes: each worker runs
``oracle.moe.moe_forward`` with ``resident`` marking its shard (pairs of other
experts contribute zero there) and the shards' outputs add up to the full
forward.  The planes come from the seeded generators in ``workloads`` (the
same draws the GPU side uploads), regenerated here per expert on access, so a
worker never holds more than one expert's planes.

Imports neither torch nor the CUDA binding: the pool is started with the
``spawn`` method and its workers only ever run CPU code.
"""
from __future__ import annotations

import numpy as np

import workloads as W
from oracle import moe as omoe


class _PerExpert:
    """``obj[e]`` draws part ``part`` of expert e's matrix (one matrix cached)."""

    def __init__(self, draw, part):
        self.draw, self.part = draw, part

    def __getitem__(self, e):
        return self.draw(int(e))[self.part]


def _cached(fn):
    memo = {}

    def get(e):
        if e not in memo:
            memo.clear()
            memo[e] = fn(e)
        return memo[e]
    return get


def plane_set(seed, fc, N, K, E, heavy):
    draw = _cached(lambda e: W.draw_plane_matrix(seed, e, fc, N, K, heavy))
    return dict(sign=_PerExpert(draw, 0), mag=_PerExpert(draw, 1), s16=_PerExpert(draw, 2),
                scale_2=W.draw_plane_scale2(seed, fc, E, K))


def delta_set(seed, fc, N, K):
    draw = _cached(lambda s: W.draw_delta_matrix(seed, s, fc, N, K))
    return dict(codes=_PerExpert(draw, 0), s4=_PerExpert(draw, 1))


def shard_forward(job):
    """y [n, H] fp64: the oracle forward of the sampled tokens restricted to ``experts``."""
    seed, H, I, E, heavy, x, idx, w, gate, slot, experts = job
    resident = np.zeros(E, dtype=bool)
    resident[np.asarray(experts, dtype=np.int64)] = True
    fc1 = plane_set(seed, 1, 2 * I, H, E, heavy)
    fc2 = plane_set(seed, 2, H, I, E, heavy)
    kw = {}
    if slot is not None:
        kw = dict(delta_slot=slot, dfc1=delta_set(seed, 1, 2 * I, H), dfc2=delta_set(seed, 2, H, I),
                  gate=gate)
    return omoe.moe_forward(x, idx, w, fc1, fc2, resident=resident, **kw)
