"""moet_moe_forward_static: the forward for callers that cannot allocate device memory.

Such callers (a plug-in handed only its input and output buffers, code running
inside a runtime whose device allocator belongs to someone else) cannot provide
the forward's workspace.  The static entry point uses a fixed scratch array in
the library's device image instead.  Checked here through the C ABI against the
workspace entry point on the same inputs, bit for bit (both run the same
deterministic kernels): before each checked call the shared scratch is filled
by a static call on unrelated data (another token count, top-k, routing, and
the delta table with a gate mask), so a kernel that read a scratch word before
writing it would see the leftovers; each check runs twice in a row, with and
without the delta.  The decode engine's shape (I = 256) and the mma.sync
engine's (I = 384) both fit the fixed scratch.  Plus the size rejection (the
binding's copy of the size is checked against the header on the CPU, in test_abi).  This
file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
H, E, SEED = 1024, 16, 77


@pytest.fixture(scope="module")
def moet():
    import __graft_entry__ as g
    g.build()
    import bit_moe_expert_moet_gb300 as m
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _layer(moet, I, dset):
    """Planes of E experts and a delta pool of len(dset) slots from the seeded generators."""
    planes, pools = {}, {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        p = [W.draw_plane_matrix(SEED + I, e, f, N, K) for e in range(E)]
        planes[f] = moet.Planes(_dev(np.stack([a[0] for a in p]).view(np.int32)),
                                _dev(np.stack([a[1] for a in p]).view(np.int32)),
                                _dev(np.stack([a[2] for a in p])),
                                _dev(W.draw_plane_scale2(SEED + I, f, E, K)))
        d = [W.draw_delta_matrix(SEED + I, s, f, N, K) for s in range(len(dset))]
        pools[f] = moet.DeltaPool(_dev(np.stack([a[0] for a in d])), _dev(np.stack([a[1] for a in d])))
    return planes, pools


class _Batch:
    """One routed batch of T tokens (top-k on device) with a gate mask."""

    def __init__(self, moet, rng, T, k):
        self.T, self.k = T, k
        self.x = _dev(W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).view(np.int16)).view(
            torch.bfloat16)
        self.idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
        self.w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        self.off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        self.perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
        moet.route_topk(_dev(rng.standard_normal((T, E)).astype(np.float32)), k, self.idx, self.w, self.off,
                        self.perm)
        self.gate = _dev((rng.random(T) < 0.5).astype(np.uint8))

    def args(self):
        return self.x, self.idx, self.w, self.off, self.perm


@pytest.mark.parametrize("I", [256, 384], ids=["decode_engine", "mma_sync_engine"])
def test_static_scratch_forward_equals_workspace_forward(moet, I):
    rng = np.random.default_rng(SEED + I)
    dset = np.array([1, 4, 9, 12], dtype=np.int32)
    planes, pools = _layer(moet, I, dset)
    slot = _dev(W.delta_slot_table(E, dset))
    dkw = dict(delta_slot=slot, dfc1=pools[1], dfc2=pools[2])
    main = _Batch(moet, rng, 9, 4)
    other = [_Batch(moet, rng, 5, 2), _Batch(moet, rng, 13, 6)]

    refs = {}
    for with_delta in (True, False):
        y = torch.empty((main.T, H), dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(moet.forward_workspace_size(main.T, H, I, E, main.k), dtype=torch.uint8, device=DEV)
        kw = dict(dkw, gate_mask=main.gate) if with_delta else {}
        moet.moe_forward(*main.args(), planes[1], planes[2], y, ws, **kw)
        refs[with_delta] = y
    torch.cuda.synchronize()
    assert moet.last_device_error() == 0

    for n, with_delta in enumerate((True, False, True)):
        # unrelated data first: the scratch now holds another batch's headers, work items,
        # activation terms, h and o
        ob = other[n % 2]
        junk = torch.empty((ob.T, H), dtype=torch.bfloat16, device=DEV)
        moet.moe_forward_static(*ob.args(), planes[1], planes[2], junk, **dict(dkw, gate_mask=ob.gate))
        for _ in range(2):                        # two calls in a row
            y = torch.full((main.T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
            kw = dict(dkw, gate_mask=main.gate) if with_delta else {}
            moet.moe_forward_static(*main.args(), planes[1], planes[2], y, **kw)
            torch.cuda.synchronize()
            assert torch.equal(y, refs[with_delta]), (I, with_delta)
    assert moet.last_device_error() == 0


def test_static_scratch_forward_rejects_oversized_layers(moet):
    lib = moet.lib
    T, H_, I, E_, k = 64, 7168, 2048, 256, 8                # needs far more than the fixed scratch
    assert moet.forward_workspace_size(T, H_, I, E_, k) > moet.FORWARD_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    p = ctypes.c_void_p(dummy.data_ptr())
    planes = moet._lib._Planes(p, p, p, p)
    status = lib.moet_moe_forward_static(T, H_, I, E_, k, p, p, p, p, p, ctypes.byref(planes),
                                         ctypes.byref(planes), None, 0, None, None, None, p, None)
    assert moet.status_string(status) == "MOET_ERR_WORKSPACE"
