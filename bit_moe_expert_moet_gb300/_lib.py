"""ctypes binding of libmoet.so: argument checks and marshalling, nothing else."""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libmoet.so")

if not os.path.exists(lib_path):
    raise ImportError(
        f"{lib_path} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()'); there is no CPU fallback")

lib = ctypes.CDLL(lib_path)

_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


class _Planes(ctypes.Structure):
    _fields_ = [("sign", _p), ("mag", _p), ("s16", _p), ("scale_2", _p)]


class _Nvfp4(ctypes.Structure):
    _fields_ = [("codes", _p), ("s4", _p)]


lib.moet_status_string.restype = ctypes.c_char_p
lib.moet_status_string.argtypes = [_i]
lib.moet_last_device_error.restype = _i
lib.moet_last_device_error.argtypes = [_p]
lib.moet_quantize_nvfp4.restype = _i
lib.moet_quantize_nvfp4.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p]
lib.moet_requant_2bit.restype = _i
lib.moet_requant_2bit.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p]
lib.moet_route_topk.restype = _i
lib.moet_route_topk.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p, _p]
lib.moet_forward_workspace_size.restype = _sz
lib.moet_forward_workspace_size.argtypes = [_i, _i, _i, _i, _i]
lib.moet_moe_forward_static.restype = _i
lib.moet_moe_forward_static.argtypes = [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p,
                                        ctypes.POINTER(_Planes), ctypes.POINTER(_Planes),
                                        _p, _i, ctypes.POINTER(_Nvfp4), ctypes.POINTER(_Nvfp4),
                                        _p, _p, _p]
FORWARD_STATIC_SCRATCH_BYTES = 8 << 20
lib.moet_debug_wait_expiry.restype = _i
lib.moet_debug_wait_expiry.argtypes = [_i, _i]
lib.moet_profile_enable.restype = _i
lib.moet_profile_enable.argtypes = [_i]
lib.moet_profile_read.restype = _i
lib.moet_profile_read.argtypes = [ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(ctypes.c_float)]
lib.moet_moe_forward.restype = _i
lib.moet_moe_forward.argtypes = [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p,
                                 ctypes.POINTER(_Planes), ctypes.POINTER(_Planes),
                                 _p, _i, ctypes.POINTER(_Nvfp4), ctypes.POINTER(_Nvfp4),
                                 _p, _p, _p, _sz, _p]
lib.moet_requant_fp8_2bit.restype = _i
lib.moet_requant_fp8_2bit.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p]
lib.moet_requant_mxfp4_2bit.restype = _i
lib.moet_sign_bias_probe.restype = _i
lib.moet_sign_bias_probe.argtypes = [_i, _i, _i, _p, ctypes.POINTER(ctypes.c_int32), _p, _p, _p]
lib.moet_requant_mxfp4_2bit.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p]
lib.moet_gate_from_confidence.restype = _i
lib.moet_gate_from_confidence.argtypes = [_i, _i, _i, _p, ctypes.c_float, _p, _p, _p, _p, _p, _p]
lib.moet_moe_forward_pooled.restype = _i
lib.moet_moe_forward_pooled.argtypes = [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _i,
                                        ctypes.POINTER(_Planes), ctypes.POINTER(_Planes),
                                        _p, _i, ctypes.POINTER(_Nvfp4), ctypes.POINTER(_Nvfp4),
                                        _p, _p, _p, _p, _p, _sz, _p]


class MoetError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)}")
        self.status = status


def status_string(status: int) -> str:
    return lib.moet_status_string(status).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise MoetError(fn, status)


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


KERNEL_KINDS = ("requant", "quantize", "route", "prologue", "fc1", "fc2", "combine", "terms", "probe")


def debug_wait_expiry(polls: int = 0, withhold: bool = False):
    """Test control of the tcgen05 engines' bounded waits (moet_debug_wait_expiry): polls > 0
    lowers the poll bound, withhold makes CTA 0 of each engine launch skip its first unit record
    so that the waits on it run out.  debug_wait_expiry() restores the defaults."""
    _check("moet_debug_wait_expiry", lib.moet_debug_wait_expiry(int(polls), 1 if withhold else 0))


def profile_enable(on: bool = True):
    _check("moet_profile_enable", lib.moet_profile_enable(1 if on else 0))


def profile_read() -> dict:
    """{kind: (launches, timed launches, summed ms)} since the previous read."""
    n = len(KERNEL_KINDS)
    la, ti, ms = (_i * n)(), (_i * n)(), (ctypes.c_float * n)()
    _check("moet_profile_read", lib.moet_profile_read(la, ti, ms))
    return {KERNEL_KINDS[i]: (la[i], ti[i], ms[i]) for i in range(n)}


def last_device_error(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise and return (and clear) the first device-side problem (0 = none)."""
    return lib.moet_last_device_error(_stream(stream))


@dataclasses.dataclass
class Planes:
    """2-bit planes of E experts of [N, K]: sign/mag int32 [E, N, K/32], s16 uint8 [E, N, K/16], scale_2 fp32 [E]."""
    sign: torch.Tensor
    mag: torch.Tensor
    s16: torch.Tensor
    scale_2: torch.Tensor

    def _c(self, name):
        return _Planes(_ptr(self.sign, torch.int32, name + ".sign"), _ptr(self.mag, torch.int32, name + ".mag"),
                       _ptr(self.s16, torch.uint8, name + ".s16"), _ptr(self.scale_2, torch.float32, name + ".scale_2"))


@dataclasses.dataclass
class DeltaPool:
    """NVFP4 delta pool of S slots of [N, K]: codes uint8 [S, N, K/2], s4 uint8 [S, N, K/16]."""
    codes: torch.Tensor
    s4: torch.Tensor

    def _c(self, name):
        return _Nvfp4(_ptr(self.codes, torch.uint8, name + ".codes"), _ptr(self.s4, torch.uint8, name + ".s4"))


def quantize_nvfp4(w: torch.Tensor, codes: torch.Tensor, s4: torch.Tensor, scale_2: torch.Tensor,
                   stream=None):
    """w fp32 [M, N, K] -> codes uint8 [M, N, K/2], s4 uint8 [M, N, K/16], scale_2 fp32 [M]."""
    M, N, K = w.shape
    _check("moet_quantize_nvfp4", lib.moet_quantize_nvfp4(
        M, N, K, _ptr(w, torch.float32, "w"), _ptr(scale_2, torch.float32, "scale_2"),
        _ptr(codes, torch.uint8, "codes"), _ptr(s4, torch.uint8, "s4"), _stream(stream)))


def requant_2bit(codes: torch.Tensor, s4: torch.Tensor, sign: torch.Tensor, mag: torch.Tensor,
                 s16: torch.Tensor, dcodes: Optional[torch.Tensor] = None, ds4: Optional[torch.Tensor] = None,
                 stream=None):
    """codes uint8 [M, N, K/2], s4 [M, N, K/16] -> sign/mag int32 [M, N, K/32], s16 [M, N, K/16] (+ delta)."""
    M, N, K2 = codes.shape
    _check("moet_requant_2bit", lib.moet_requant_2bit(
        M, N, 2 * K2, _ptr(codes, torch.uint8, "codes"), _ptr(s4, torch.uint8, "s4"),
        _ptr(sign, torch.int32, "sign"), _ptr(mag, torch.int32, "mag"), _ptr(s16, torch.uint8, "s16"),
        _ptr(dcodes, torch.uint8, "dcodes"), _ptr(ds4, torch.uint8, "ds4"), _stream(stream)))


def route_topk(logits: torch.Tensor, k: int, topk_idx: torch.Tensor, topk_w: torch.Tensor,
               expert_offsets: torch.Tensor, perm: torch.Tensor, stream=None):
    T, E = logits.shape
    _check("moet_route_topk", lib.moet_route_topk(
        T, E, k, _ptr(logits, torch.float32, "logits"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(expert_offsets, torch.int32, "expert_offsets"),
        _ptr(perm, torch.int32, "perm"), _stream(stream)))


def forward_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib.moet_forward_workspace_size(T, H, I, E, k))


def moe_forward(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                expert_offsets: torch.Tensor, perm: torch.Tensor, fc1: Planes, fc2: Planes,
                y: torch.Tensor, workspace: torch.Tensor, delta_slot: Optional[torch.Tensor] = None,
                dfc1: Optional[DeltaPool] = None, dfc2: Optional[DeltaPool] = None,
                gate_mask: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [T, H] -> y bf16 [T, H] (written).  fc1 planes [E, 2I, H/..], fc2 [E, H, I/..]."""
    T, H = x.shape
    E = fc1.scale_2.shape[0]
    I = fc2.sign.shape[2] * 32
    k = topk_idx.shape[1]
    if x.dtype != torch.bfloat16 or y.dtype != torch.bfloat16:
        raise TypeError("x and y must be bfloat16")
    c1, c2 = fc1._c("fc1"), fc2._c("fc2")
    n_slots = 0
    d1 = d2 = None
    if delta_slot is not None:
        if dfc1 is None or dfc2 is None or gate_mask is None:
            raise ValueError("delta_slot needs dfc1, dfc2 and gate_mask")
        n_slots = dfc1.codes.shape[0]
        d1, d2 = dfc1._c("dfc1"), dfc2._c("dfc2")
    _check("moet_moe_forward", lib.moet_moe_forward(
        T, H, I, E, k, _ptr(x, None, "x"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(expert_offsets, torch.int32, "expert_offsets"),
        _ptr(perm, torch.int32, "perm"), ctypes.byref(c1), ctypes.byref(c2),
        _ptr(delta_slot, torch.int32, "delta_slot"), n_slots,
        ctypes.byref(d1) if d1 is not None else None, ctypes.byref(d2) if d2 is not None else None,
        _ptr(gate_mask, torch.uint8, "gate_mask"), _ptr(y, None, "y"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def requant_fp8_2bit(codes: torch.Tensor, bscale: torch.Tensor, scale_2: torch.Tensor, sign: torch.Tensor,
                     mag: torch.Tensor, s16: torch.Tensor, dcodes: Optional[torch.Tensor] = None,
                     ds4: Optional[torch.Tensor] = None, stream=None):
    """FP8 block-quant codes u8 [M, N, K] with fp32 128x128 block scales [M, ceil(N/128), ceil(K/128)]
    -> scale_2 fp32 [M], planes and s16 (+ delta codes/scales), all written."""
    M, N, K = codes.shape
    _check("moet_requant_fp8_2bit", lib.moet_requant_fp8_2bit(
        M, N, K, _ptr(codes, torch.uint8, "codes"), _ptr(bscale, torch.float32, "bscale"),
        _ptr(scale_2, torch.float32, "scale_2"), _ptr(sign, torch.int32, "sign"), _ptr(mag, torch.int32, "mag"),
        _ptr(s16, torch.uint8, "s16"), _ptr(dcodes, torch.uint8, "dcodes"), _ptr(ds4, torch.uint8, "ds4"),
        _stream(stream)))


def requant_mxfp4_2bit(codes: torch.Tensor, e8m0: torch.Tensor, scale_2: torch.Tensor, sign: torch.Tensor,
                       mag: torch.Tensor, s16: torch.Tensor, dcodes: Optional[torch.Tensor] = None,
                       ds4: Optional[torch.Tensor] = None, stream=None):
    """MXFP4 codes u8 [M, N, K/2] with E8M0 scales u8 [M, N, K/32] -> scale_2 fp32 [M], planes and
    s16 (+ delta codes/scales), all written."""
    M, N, K2 = codes.shape
    _check("moet_requant_mxfp4_2bit", lib.moet_requant_mxfp4_2bit(
        M, N, 2 * K2, _ptr(codes, torch.uint8, "codes"), _ptr(e8m0, torch.uint8, "e8m0"),
        _ptr(scale_2, torch.float32, "scale_2"), _ptr(sign, torch.int32, "sign"), _ptr(mag, torch.int32, "mag"),
        _ptr(s16, torch.uint8, "s16"), _ptr(dcodes, torch.uint8, "dcodes"), _ptr(ds4, torch.uint8, "ds4"),
        _stream(stream)))


def sign_bias_probe(w: torch.Tensor, levels, row_sums: torch.Tensor, sums: torch.Tensor, stream=None):
    """fp32 weights [M, N, K] and 4 ascending integer levels -> per-row fp64 sums [M, N, 4] and
    per-matrix sums [M, 4] of W, W^2, Q - W and (Q - W)^2 for the per-block L2-optimal fit."""
    M, N, K = w.shape
    lv = (ctypes.c_int32 * 4)(*[int(v) for v in levels])
    _check("moet_sign_bias_probe", lib.moet_sign_bias_probe(
        M, N, K, _ptr(w, torch.float32, "w"), lv, _ptr(row_sums, torch.float64, "row_sums"),
        _ptr(sums, torch.float64, "sums"), _stream(stream)))


def gate_from_confidence(conf: torch.Tensor, tau: float, topk_idx: torch.Tensor, gate_mask: torch.Tensor,
                         delta_slot: Optional[torch.Tensor] = None, need_mask: Optional[torch.Tensor] = None,
                         counts: Optional[torch.Tensor] = None, n_experts: Optional[int] = None, stream=None):
    """gate_mask[t] = conf[t] < tau (u8); need_mask[e] = 1 for experts a gated token routes to that
    have no delta slot; counts (int32 [2]) += (gated tokens, such pairs)."""
    T, k = topk_idx.shape
    E = n_experts if n_experts is not None else (delta_slot.shape[0] if delta_slot is not None else
                                                 (need_mask.shape[0] if need_mask is not None else None))
    if E is None:
        raise ValueError("n_experts is needed without delta_slot or need_mask")
    if counts is not None and (counts.dtype != torch.int32 or counts.numel() < 2):
        raise TypeError("counts must be an int32 tensor of at least two elements (u32 counters)")
    _check("moet_gate_from_confidence", lib.moet_gate_from_confidence(
        T, E, k, _ptr(conf, torch.float32, "conf"), float(tau), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(delta_slot, torch.int32, "delta_slot"), _ptr(gate_mask, torch.uint8, "gate_mask"),
        _ptr(need_mask, torch.uint8, "need_mask"), _ptr(counts, None, "counts"), _stream(stream)))


def moe_forward_pooled(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                       expert_offsets: torch.Tensor, perm: torch.Tensor, expert_slot: torch.Tensor,
                       fc1: Planes, fc2: Planes, y: torch.Tensor, workspace: torch.Tensor,
                       delta_slot: Optional[torch.Tensor] = None, dfc1: Optional[DeltaPool] = None,
                       dfc2: Optional[DeltaPool] = None, gate_mask: Optional[torch.Tensor] = None,
                       miss_count: Optional[torch.Tensor] = None, miss_mask: Optional[torch.Tensor] = None,
                       stream=None):
    """moe_forward over a pool of resident experts: fc1/fc2 hold n_pool slots, expert e lives in
    slot expert_slot[e] (-1 = not resident: contributes zero, counted in miss_count (u32 [1]) and
    flagged in miss_mask (u8 [E]))."""
    T, H = x.shape
    E = expert_slot.shape[0]
    n_pool = fc1.scale_2.shape[0]
    I = fc2.sign.shape[2] * 32
    k = topk_idx.shape[1]
    if x.dtype != torch.bfloat16 or y.dtype != torch.bfloat16:
        raise TypeError("x and y must be bfloat16")
    if miss_count is not None and (miss_count.dtype != torch.int32 or miss_count.numel() < 1):
        raise TypeError("miss_count must be an int32 tensor of at least one element (the u32 counter)")
    c1, c2 = fc1._c("fc1"), fc2._c("fc2")
    n_slots = 0
    d1 = d2 = None
    if delta_slot is not None:
        if dfc1 is None or dfc2 is None or gate_mask is None:
            raise ValueError("delta_slot needs dfc1, dfc2 and gate_mask")
        n_slots = dfc1.codes.shape[0]
        d1, d2 = dfc1._c("dfc1"), dfc2._c("dfc2")
    _check("moet_moe_forward_pooled", lib.moet_moe_forward_pooled(
        T, H, I, E, k, _ptr(x, None, "x"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(expert_offsets, torch.int32, "expert_offsets"),
        _ptr(perm, torch.int32, "perm"), _ptr(expert_slot, torch.int32, "expert_slot"), n_pool,
        ctypes.byref(c1), ctypes.byref(c2),
        _ptr(delta_slot, torch.int32, "delta_slot"), n_slots,
        ctypes.byref(d1) if d1 is not None else None, ctypes.byref(d2) if d2 is not None else None,
        _ptr(gate_mask, torch.uint8, "gate_mask"), _ptr(miss_count, None, "miss_count"),
        _ptr(miss_mask, torch.uint8, "miss_mask"), _ptr(y, None, "y"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_forward_static(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                       expert_offsets: torch.Tensor, perm: torch.Tensor, fc1: Planes, fc2: Planes,
                       y: torch.Tensor, delta_slot: Optional[torch.Tensor] = None,
                       dfc1: Optional[DeltaPool] = None, dfc2: Optional[DeltaPool] = None,
                       gate_mask: Optional[torch.Tensor] = None, stream=None):
    """moe_forward without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 8 MiB array inside the library's device image
    (shared by all calls; overlapping calls must be serialised by the caller)."""
    T, H = x.shape
    E = fc1.scale_2.shape[0]
    I = fc2.sign.shape[2] * 32
    k = topk_idx.shape[1]
    if x.dtype != torch.bfloat16 or y.dtype != torch.bfloat16:
        raise TypeError("x and y must be bfloat16")
    c1, c2 = fc1._c("fc1"), fc2._c("fc2")
    n_slots = 0
    d1 = d2 = None
    if delta_slot is not None:
        if dfc1 is None or dfc2 is None or gate_mask is None:
            raise ValueError("delta_slot needs dfc1, dfc2 and gate_mask")
        n_slots = dfc1.codes.shape[0]
        d1, d2 = dfc1._c("dfc1"), dfc2._c("dfc2")
    _check("moet_moe_forward_static", lib.moet_moe_forward_static(
        T, H, I, E, k, _ptr(x, None, "x"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(expert_offsets, torch.int32, "expert_offsets"),
        _ptr(perm, torch.int32, "perm"), ctypes.byref(c1), ctypes.byref(c2),
        _ptr(delta_slot, torch.int32, "delta_slot"), n_slots,
        ctypes.byref(d1) if d1 is not None else None, ctypes.byref(d2) if d2 is not None else None,
        _ptr(gate_mask, torch.uint8, "gate_mask"), _ptr(y, None, "y"), _stream(stream)))
