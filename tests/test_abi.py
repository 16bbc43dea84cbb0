"""The C ABI library loads, exports every symbol include/moet.h declares, and its
host-side argument checks reject bad calls before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from bit_moe_expert_moet_gb300 import _lib
    return _lib.lib


def _declared():
    with open(os.path.join(ROOT, "include", "moet.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moet_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("moet_requant_2bit", "moet_route_topk", "moet_moe_forward",
                     "moet_forward_workspace_size", "moet_status_string", "moet_last_device_error",
                     "moet_quantize_nvfp4"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(9):
        assert lib.moet_status_string(code).decode().startswith("MOET_")
    assert lib.moet_status_string(99).decode() == "MOET_ERR_UNKNOWN"


def test_host_side_rejections(lib):
    # shape checks come first and return before any CUDA call
    assert lib.moet_route_topk(0, 8, 2, None, None, None, None, None, None) == 2          # SHAPE
    assert lib.moet_route_topk(4, 2048, 2, None, None, None, None, None, None) == 2       # E > 1024
    assert lib.moet_route_topk(4, 8, 17, None, None, None, None, None, None) == 2         # k > 16
    assert lib.moet_route_topk(4, 8, 2, None, None, None, None, None, None) == 1          # null -> INVALID_ARG
    assert lib.moet_requant_2bit(1, 1, 48, None, None, None, None, None, None, None, None) == 2   # K % 32
    assert lib.moet_requant_2bit(1, 1, 64, None, None, None, None, None, None, None, None) == 1
    p = ctypes.c_void_p(16)                                                               # aligned dummy
    q = ctypes.c_void_p(17)                                                               # misaligned
    assert lib.moet_requant_2bit(1, 1, 64, q, p, p, p, p, None, None, None) == 3          # ALIGN
    assert lib.moet_requant_2bit(1, 1, 64, p, p, p, p, p, p, None, None) == 1             # half a delta
    assert lib.moet_quantize_nvfp4(1, 1, 40, p, p, p, p, None) == 2
    fwd_null = [None] * 8 + [0] + [None] * 5 + [0, None]
    assert lib.moet_moe_forward(1, 100, 128, 8, 2, *fwd_null) == 2                         # H % 128
    assert lib.moet_moe_forward(1, 128, 128, 8, 2, *fwd_null) == 1                         # nulls


def test_host_side_rejections_of_the_load_time_and_cache_calls(lib):
    """FP8 / MXFP4 requant, the sign-bias probe, the confidence gate and the pooled forward reject
    bad shapes, null pointers, misaligned buffers and bad codebooks before any CUDA call."""
    p = ctypes.c_void_p(256)                                                              # aligned dummy
    q = ctypes.c_void_p(258)                                                              # misaligned
    for fn in (lib.moet_requant_fp8_2bit, lib.moet_requant_mxfp4_2bit):
        assert fn(0, 4, 64, p, p, p, p, p, p, None, None, None) == 2                      # M < 1
        assert fn(1, 4, 48, p, p, p, p, p, p, None, None, None) == 2                      # K % 32
        assert fn(1, 4, 64, None, p, p, p, p, p, None, None, None) == 1                   # null codes
        assert fn(1, 4, 64, p, p, p, p, p, p, p, None, None) == 1                         # half a delta
        assert fn(1, 4, 64, q, p, p, p, p, p, None, None, None) == 3                      # codes not 16 B
    lv = lambda *v: (ctypes.c_int32 * 4)(*v)
    probe = lib.moet_sign_bias_probe
    assert probe(1, 4, 40, p, lv(-2, -1, 0, 1), p, p, None) == 2                          # K % 16
    assert probe(1, 4, 64, None, lv(-2, -1, 0, 1), p, p, None) == 1                       # null weights
    assert probe(1, 4, 64, p, lv(-1, -1, 0, 1), p, p, None) == 1                          # not ascending
    assert probe(1, 4, 64, p, lv(-65, -1, 1, 3), p, p, None) == 1                         # out of range
    assert probe(1, 4, 64, q, lv(-2, -1, 0, 1), p, p, None) == 3                          # w not 16 B
    gate = lib.moet_gate_from_confidence
    assert gate(4, 8, 9, p, 0.6, p, None, p, None, None, None) == 2                       # k > E
    assert gate(4, 2048, 2, p, 0.6, p, None, p, None, None, None) == 2                    # E > 1024
    assert gate(4, 8, 2, None, 0.6, p, None, p, None, None, None) == 1                    # null conf
    assert gate(4, 8, 2, ctypes.c_void_p(257), 0.6, p, None, p, None, None, None) == 3    # conf not 4 B
    pooled = lib.moet_moe_forward_pooled
    # fc1, fc2, delta_slot, n_slots, dfc1, dfc2, gate_mask, miss_count, miss_mask, y, workspace, bytes, stream
    tail = [None, None, None, 0, None, None, None, None, None, None, None, 0, None]
    assert pooled(1, 128, 128, 8, 2, p, p, p, p, p, None, 4, *tail) == 1                  # null slot table
    assert pooled(1, 128, 128, 8, 2, p, p, p, p, p, p, 0, *tail) == 2                     # empty pool
    assert pooled(1, 128, 128, 8, 2, p, p, p, p, p, ctypes.c_void_p(258), 4, *tail) == 3  # slot table not 4 B


def test_static_forward_rejects_layers_larger_than_its_scratch(lib):
    """moet_moe_forward_static checks the layer against its fixed 8 MiB scratch before any CUDA
    call: the DeepSeek-V3 decode layer fits up to T = 13 tokens (as the header states) and is
    rejected beyond."""
    import bit_moe_expert_moet_gb300 as m
    ws = lib.moet_forward_workspace_size
    assert ws(13, 7168, 2048, 256, 8) <= m.FORWARD_STATIC_SCRATCH_BYTES < ws(14, 7168, 2048, 256, 8)
    nulls = [None] * 5 + [None, None, None, 0, None, None, None, None, None]
    assert lib.moet_moe_forward_static(14, 7168, 2048, 256, 8, *nulls) == 5               # WORKSPACE
    assert lib.moet_moe_forward_static(0, 7168, 2048, 256, 8, *nulls) == 2                # SHAPE


def test_workspace_size_is_monotone(lib):
    ws = lib.moet_forward_workspace_size
    a = ws(1, 7168, 2048, 256, 8)
    b = ws(64, 7168, 2048, 256, 8)
    assert 0 < a < b
    assert ws(0, 7168, 2048, 256, 8) == 0
    # fp32 h [T k, I] and o [T k, H] dominate
    assert b >= 64 * 8 * (7168 + 2048) * 4


def test_static_scratch_size_matches_header(lib):
    """The binding's copy of the fixed scratch size of moet_moe_forward_static is the header's."""
    from bit_moe_expert_moet_gb300 import _lib
    with open(os.path.join(ROOT, "include", "moet.h")) as f:
        m = re.search(r"#define\s+MOET_FORWARD_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", f.read())
    assert m is not None
    assert _lib.FORWARD_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_debug_wait_expiry_rejects_bad_arguments(lib):
    assert lib.moet_debug_wait_expiry(-1, 0) == 1          # INVALID_ARG, nothing copied
    assert lib.moet_debug_wait_expiry(0, 2) == 1
