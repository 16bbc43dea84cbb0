"""moet_moe_forward_static: the forward for callers that cannot allocate device memory.

Such callers (a plug-in handed only its input and output buffers, code running
inside a runtime whose device allocator belongs to someone else) cannot provide
the forward's workspace.  The static entry point uses a fixed scratch array in
the library's device image instead.  Checked here through the C ABI against the
workspace entry point on the same inputs, for two calls in a row (the second
call finds the first call's leftovers in the shared scratch), plus the size
rejection.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from oracle import nvfp4 as onv, requant as orq

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL_FROB, MAX_ABS = 5e-3, 2e-2


@pytest.fixture(scope="module")
def moet():
    import __graft_entry__ as g
    g.build()
    import bit_moe_expert_moet_gb300 as m
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _layer(moet, H, I, E, rng):
    planes = {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
        q = [onv.quantize(w[e]) for e in range(E)]
        rq = [orq.requant_2bit(a[0], a[1], want_delta=False) for a in q]
        planes[f] = moet.Planes(_dev(np.stack([r["sign"] for r in rq]).view(np.int32)),
                                _dev(np.stack([r["mag"] for r in rq]).view(np.int32)),
                                _dev(np.stack([r["s16"] for r in rq])),
                                _dev(np.array([a[2] for a in q], np.float32)))
    return planes


def _close(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    mx = np.abs(a - b).max() / np.sqrt(np.mean(b ** 2))
    return rel <= REL_FROB and mx <= MAX_ABS, (rel, mx)


def test_static_scratch_forward_matches_workspace_forward(moet):
    H, I, E, k, T = 1024, 256, 16, 4, 9
    rng = np.random.default_rng(77)
    planes = _layer(moet, H, I, E, rng)
    logits = _dev(rng.standard_normal((T, E)).astype(np.float32))
    x = _dev(W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).view(np.int16)).view(torch.bfloat16)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(logits, k, idx, w, off, perm)
    y_ref = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    moet.moe_forward(x, idx, w, off, perm, planes[1], planes[2], y_ref, ws)
    ref = y_ref.float().cpu().numpy()
    outs = []
    for _ in range(2):
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moet.moe_forward_static(x, idx, w, off, perm, planes[1], planes[2], y)
        torch.cuda.synchronize()
        outs.append(y.float().cpu().numpy())
    assert moet.last_device_error() == 0
    for o in outs:
        ok, err = _close(o, ref)
        assert ok, err


def test_static_scratch_forward_rejects_oversized_layers(moet):
    lib = moet.lib
    T, H, I, E, k = 64, 7168, 2048, 256, 8                # needs far more than the fixed scratch
    assert moet.forward_workspace_size(T, H, I, E, k) > moet.FORWARD_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    p = ctypes.c_void_p(dummy.data_ptr())
    planes = moet._lib._Planes(p, p, p, p)
    status = lib.moet_moe_forward_static(T, H, I, E, k, p, p, p, p, p, ctypes.byref(planes),
                                         ctypes.byref(planes), None, 0, None, None, None, p, None)
    assert moet.status_string(status) == "MOET_ERR_WORKSPACE"
