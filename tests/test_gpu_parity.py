"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Integer outputs (NVFP4 codes/scales, planes, s16, delta, top-k ids, offsets,
permutation) must match bit for bit; routing weights within 1e-6; the layer
output within relative Frobenius 5e-3 and max-abs 2e-2 rms(y*) (the bound and
when the bf16 rounding of the exact output is taken out of it: ``_parity``).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import gate as ogate, moe as omoe, nvfp4 as onv, requant as orq, route as oroute
from _parity import check_y

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def moet():
    import __graft_entry__ as g
    g.build()
    import bit_moe_expert_moet_gb300 as m
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.cpu().numpy()


# ------------------------------------------------------------------ quantiser / requant
def _gpu_quantize(moet, w):
    M, N, K = w.shape
    codes = torch.empty((M, N, K // 2), dtype=torch.uint8, device=DEV)
    s4 = torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV)
    sc2 = torch.empty(M, dtype=torch.float32, device=DEV)
    moet.quantize_nvfp4(dev(w), codes, s4, sc2)
    return host(codes), host(s4), host(sc2)


def _gpu_requant(moet, codes, s4, delta=True):
    M, N, K2 = codes.shape
    K = 2 * K2
    sign = torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV)
    mag = torch.empty_like(sign)
    s16 = torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV)
    dc = torch.empty((M, N, K // 2), dtype=torch.uint8, device=DEV) if delta else None
    ds = torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV) if delta else None
    moet.requant_2bit(dev(codes), dev(s4), sign, mag, s16, dc, ds)
    out = dict(sign=host(sign).view(np.uint32), mag=host(mag).view(np.uint32), s16=host(s16))
    if delta:
        out["dcodes"], out["ds4"] = host(dc), host(ds)
    return out


def test_quantize_nvfp4_bit_exact(moet):
    rng = np.random.default_rng(20)
    ws = [
        (rng.standard_normal((64, 256)) * 0.02).astype(np.float32),
        (rng.standard_t(4, (64, 256)) * 0.014).astype(np.float32),
        (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-40, 40, (64, 1)))).astype(np.float32),
        np.zeros((64, 256), np.float32),
    ]
    ws[0][3, 16:32] = 0.0
    ws[0][5, :16] = -0.0
    ws[1][7, 40] = 1e-30
    w = np.stack(ws)
    codes, s4, sc2 = _gpu_quantize(moet, w)
    for m in range(w.shape[0]):
        oc, os4, osc = onv.quantize(w[m])
        assert np.float32(osc) == sc2[m]
        assert np.array_equal(os4, s4[m])
        assert np.array_equal(oc, codes[m])


def _random_nvfp4(rng, M, N, K):
    codes = rng.integers(0, 256, (M, N, K // 2), dtype=np.uint8)
    codes[rng.random(codes.shape) < 0.05] = 0
    s4 = rng.integers(0, 127, (M, N, K // 16), dtype=np.uint8)
    s4[rng.random(s4.shape) < 0.03] = 0
    return codes, s4


def _check_requant(got, codes, s4):
    for m in range(codes.shape[0]):
        ref = orq.requant_2bit(codes[m], s4[m], want_delta="dcodes" in got)
        for key in ("sign", "mag", "s16", "dcodes", "ds4"):
            if key in got:
                assert np.array_equal(ref[key], got[key][m]), (m, key)


@pytest.mark.parametrize("delta", [True, False], ids=["with_delta", "planes_only"])
def test_requant_bit_exact_random(moet, delta):
    rng = np.random.default_rng(21)
    codes, s4 = _random_nvfp4(rng, 3, 64, 512)
    _check_requant(_gpu_requant(moet, codes, s4, delta), codes, s4)


@pytest.mark.parametrize("delta", [True, False], ids=["with_delta", "planes_only"])
def test_requant_exhaustive_scale_and_max_code(moet, delta):
    """Every (s4, max code) pair, including all s16 ties in the e4m3 subnormal range; the
    planes-only kernel (a table per (s4, max code) and integer bit gathers) and the delta kernel
    (the rule weight by weight) both."""
    rows = []
    rng = np.random.default_rng(22)
    for s in range(127):
        for mx in range(8):
            c = rng.integers(0, mx + 1, 32).astype(np.uint8) | (rng.integers(0, 2, 32).astype(np.uint8) << 3)
            c[0] = mx | (8 if s & 1 else 0)
            c[17] = mx
            rows.append((c, s))
    codes = np.stack([(c[0::2] | (c[1::2] << 4)).astype(np.uint8) for c, _ in rows])[None]
    s4 = np.array([[s, (s * 7 + 3) % 127] for _, s in rows], dtype=np.uint8)[None]
    _check_requant(_gpu_requant(moet, codes, s4, delta), codes, s4)


def test_requant_planes_large_ragged(moet):
    """A pass of many grid-stride iterations with a ragged tail (3 x 4099 rows x 7168): the
    planes-only kernel equals the delta kernel's planes everywhere, and sampled rows equal the
    oracle (the rule is local to a row)."""
    rng = np.random.default_rng(24)
    M, N, K = 3, 4099, 7168
    codes = rng.integers(0, 256, (M, N, K // 2), dtype=np.uint8)
    s4 = rng.integers(0, 127, (M, N, K // 16), dtype=np.uint8)
    a = _gpu_requant(moet, codes, s4, delta=True)
    b = _gpu_requant(moet, codes, s4, delta=False)
    for key in ("sign", "mag", "s16"):
        assert np.array_equal(a[key], b[key]), key
    for m in range(M):
        rows = np.unique(np.r_[0, N - 1, rng.integers(0, N, 6)])
        ref = orq.requant_2bit(codes[m, rows], s4[m, rows], want_delta=False)
        for key in ("sign", "mag", "s16"):
            assert np.array_equal(ref[key], b[key][m, rows]), (m, key)


@pytest.mark.parametrize("M,N,K,wide", [(3, 200, 96, False), (1, 128, 2048, False), (2, 7, 32, False),
                                         (2, 300, 640, True), (5, 64, 8192, True)])
def test_requant_fp8_bit_exact(moet, M, N, K, wide):
    """FP8 block-quant -> scale_2, planes, s16 and delta, bit-exact against the oracle; N and K
    not multiples of the 128 x 128 scale blocks, signed zeros, +-448 and subnormals included,
    and an all-zero matrix.  The wide cases spread the block scales over 2^-120 .. 2^20 (an fp32
    subnormal and a zero scale among them), so most blocks sit far below the matrix's largest
    and get a zero or subnormal s16; the amax pass then runs on many CTAs per matrix."""
    rng = np.random.default_rng(140 + N + K)
    codes = rng.integers(0, 256, (M, N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] ^= 1
    codes[0, 0, :5] = [0x00, 0x80, 0x7E, 0xFE, 0x01]
    if M > 1:
        codes[-1] = 0                                       # an all-zero matrix
    shape = (M, (N + 127) // 128, (K + 127) // 128)
    if wide:
        bs = np.ldexp(rng.random(shape) + 0.5, rng.integers(-120, 21, shape)).astype(np.float32)
        bs[0, 0, 0] = np.float32(3e-43)
        bs[0, -1, -1] = 0.0
        codes[0, :16, 128:144] = codes[0, 0, 128]           # sixteen equal codes in a row of a block
    else:
        bs = (rng.random(shape) * 0.02 + 0.001).astype(np.float32)
    g = dict(scale_2=torch.empty(M, dtype=torch.float32, device=DEV),
             sign=torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV),
             mag=torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV),
             s16=torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV),
             dcodes=torch.empty((M, N, K // 2), dtype=torch.uint8, device=DEV),
             ds4=torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV))
    moet.requant_fp8_2bit(dev(codes), dev(bs), g["scale_2"], g["sign"], g["mag"], g["s16"], g["dcodes"], g["ds4"])
    torch.cuda.synchronize()
    for m in range(M):
        o = orq.requant_fp8_2bit(codes[m], bs[m])
        assert host(g["scale_2"])[m] == o["scale_2"]
        assert np.array_equal(host(g["sign"])[m].view(np.uint32), o["sign"])
        assert np.array_equal(host(g["mag"])[m].view(np.uint32), o["mag"])
        for key in ("s16", "dcodes", "ds4"):
            assert np.array_equal(host(g[key])[m], o[key]), key
    # without the delta outputs: the same planes
    sign2 = torch.empty_like(g["sign"]); mag2 = torch.empty_like(g["mag"]); s162 = torch.empty_like(g["s16"])
    sc2 = torch.empty_like(g["scale_2"])
    moet.requant_fp8_2bit(dev(codes), dev(bs), sc2, sign2, mag2, s162)
    assert torch.equal(sign2, g["sign"]) and torch.equal(mag2, g["mag"]) and torch.equal(s162, g["s16"])


@pytest.mark.parametrize("M,N,K,lo,hi", [(3, 200, 96, 100, 150), (1, 128, 2048, 100, 150), (2, 7, 32, 100, 150),
                                         (4, 300, 512, 0, 255)])
def test_requant_mxfp4_bit_exact(moet, M, N, K, lo, hi):
    """MXFP4 (e2m1 codes, E8M0 scale per 32 along K) -> scale_2, planes, s16 and delta, bit-exact
    against the oracle; signed zeros, +-6, the extreme exponents 2^-127 and 2^127 in one matrix
    and an all-zero matrix included; the last case draws exponents over the whole E8M0 range."""
    rng = np.random.default_rng(150 + N + K)
    codes = rng.integers(0, 256, (M, N, K // 2), dtype=np.uint8)
    codes[0, 0, :2] = [0x80, 0x7F]
    e8m0 = rng.integers(lo, hi, (M, N, K // 32)).astype(np.uint8)
    e8m0[0, 0, 0] = 0
    e8m0[0, -1, -1] = 254
    if M > 1:
        codes[-1] = 0                                       # an all-zero matrix
    g = dict(scale_2=torch.empty(M, dtype=torch.float32, device=DEV),
             sign=torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV),
             mag=torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV),
             s16=torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV),
             dcodes=torch.empty((M, N, K // 2), dtype=torch.uint8, device=DEV),
             ds4=torch.empty((M, N, K // 16), dtype=torch.uint8, device=DEV))
    moet.requant_mxfp4_2bit(dev(codes), dev(e8m0), g["scale_2"], g["sign"], g["mag"], g["s16"], g["dcodes"],
                            g["ds4"])
    torch.cuda.synchronize()
    for m in range(M):
        o = orq.requant_mxfp4_2bit(codes[m], e8m0[m])
        assert host(g["scale_2"])[m] == o["scale_2"]
        assert np.array_equal(host(g["sign"])[m].view(np.uint32), o["sign"])
        assert np.array_equal(host(g["mag"])[m].view(np.uint32), o["mag"])
        for key in ("s16", "dcodes", "ds4"):
            assert np.array_equal(host(g[key])[m], o[key]), key
    sign2 = torch.empty_like(g["sign"]); mag2 = torch.empty_like(g["mag"]); s162 = torch.empty_like(g["s16"])
    sc2 = torch.empty_like(g["scale_2"])
    moet.requant_mxfp4_2bit(dev(codes), dev(e8m0), sc2, sign2, mag2, s162)
    assert torch.equal(sign2, g["sign"]) and torch.equal(mag2, g["mag"]) and torch.equal(s162, g["s16"])


def test_requant_without_delta_matches_planes(moet):
    rng = np.random.default_rng(23)
    codes, s4 = _random_nvfp4(rng, 2, 32, 256)
    a = _gpu_requant(moet, codes, s4, delta=True)
    b = _gpu_requant(moet, codes, s4, delta=False)
    for key in ("sign", "mag", "s16"):
        assert np.array_equal(a[key], b[key])


# ------------------------------------------------------------------ routing
def _gpu_route(moet, logits, k):
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(dev(logits), k, idx, w, off, perm)
    return host(idx), host(w), host(off), host(perm)


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (4, 8, 2), (37, 64, 6), (64, 256, 8), (512, 384, 8),
                                   (513, 256, 8), (4096, 256, 8), (256, 1024, 16), (100, 16, 1), (9, 33, 5),
                                   (700, 64, 7), (3000, 1024, 16), (16, 1024, 16), (15, 100, 15), (16, 7, 7)])
def test_route_bit_exact(moet, T, E, k):
    """Every routing path: up to 16 tokens in one CTA with the counting bucketing (at its 256-pair
    limit, with a pair count that needs padding, and with every expert chosen by every token),
    the two-kernel path up to 4096 pairs, the multi-CTA path beyond."""
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 1] = logits[:, 2]                   # ties -> lower id
    if T > 3:
        logits[2, :] = 0.25                        # all equal
        logits[3, ::3] = -np.inf
    idx, w, off, perm = _gpu_route(moet, logits, k)
    oi, ow = oroute.route_topk(logits, k)
    assert np.array_equal(idx, oi)
    assert np.abs(w - ow).max() <= 1e-6
    _, ooff, operm = oroute.bucket(oi, E)
    assert np.array_equal(off, ooff)
    assert np.array_equal(perm, operm)


def test_route_nan_ranks_below_minus_inf(moet):
    logits = np.array([[np.nan, -np.inf, 1.0, 2.0, np.nan, -0.0, 0.0, -1.0]], dtype=np.float32)
    idx, w, _, _ = _gpu_route(moet, logits, 7)
    oi, _ = oroute.route_topk(logits, 7)
    assert np.array_equal(idx, oi)
    assert idx[0].tolist() == [3, 2, 5, 6, 7, 1, 0]


# ------------------------------------------------------------------ forward
def _make_layer(moet, H, I, E, dset, rng=None, cfg=None):
    """GPU planes + delta pool from fp32 weights via the oracle quantiser (host)."""
    ref, gp = {}, {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        if cfg is not None:
            w = np.stack([W.draw_weight(cfg, e, f) for e in range(E)])
        else:
            w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
        q = [onv.quantize(w[e]) for e in range(E)]
        codes = np.stack([a[0] for a in q])
        s4 = np.stack([a[1] for a in q])
        sc2 = np.array([a[2] for a in q], np.float32)
        got = _gpu_requant(moet, codes, s4, delta=True)
        rq = [orq.requant_2bit(codes[e], s4[e]) for e in range(E)]
        for key in ("sign", "mag", "s16", "dcodes", "ds4"):
            assert np.array_equal(np.stack([r[key] for r in rq]), got[key])
        # the oracle runs on its own requant output (identical to the GPU's, checked above)
        ref[f] = dict(sign=np.stack([r["sign"] for r in rq]), mag=np.stack([r["mag"] for r in rq]),
                      s16=np.stack([r["s16"] for r in rq]), scale_2=sc2)
        ref[f, "d"] = dict(codes=np.stack([r["dcodes"] for r in rq])[dset],
                           s4=np.stack([r["ds4"] for r in rq])[dset])
        gp[f] = moet.Planes(dev(got["sign"].view(np.int32)), dev(got["mag"].view(np.int32)), dev(got["s16"]), dev(sc2))
        gp[f, "d"] = moet.DeltaPool(dev(got["dcodes"][dset]), dev(got["ds4"][dset]))
    return ref, gp


def _run_forward(moet, logits, xb, k, gp, E, H, dset=None, gate=None, slot=None):
    T = logits.shape[0]
    ld = dev(logits)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(ld, k, idx, w, off, perm)
    x = dev(xb.view(np.int16)).view(torch.bfloat16)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    I = gp[2].sign.shape[2] * 32
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    kw = {}
    if dset is not None:
        if slot is None:
            slot = W.delta_slot_table(E, dset)
        kw = dict(delta_slot=dev(slot), dfc1=gp[1, "d"], dfc2=gp[2, "d"], gate_mask=dev(gate))
    moet.moe_forward(x, idx, w, off, perm, gp[1], gp[2], y, ws, **kw)
    err = moet.last_device_error()
    return y.float().cpu().numpy(), err


def _oracle_forward(logits, xb, k, ref, dset=None, gate=None, E=None, tokens=None, slot=None):
    oi, ow = oroute.route_topk(logits, k)
    x = W.bf16_bits_to_f32(xb).astype(np.float64)
    if dset is None:
        return omoe.moe_forward(x, oi, ow, ref[1], ref[2], tokens=tokens)
    if slot is None:
        slot = W.delta_slot_table(E, dset)
    return omoe.moe_forward(x, oi, ow, ref[1], ref[2], slot, ref[1, "d"], ref[2, "d"], gate, tokens=tokens)


@pytest.mark.parametrize("gate_mode", ["config", "all"])
def test_forward_tiny_layer(moet, gate_mode):
    cfg = W.CONFIGS["tiny"]
    logits, xb, dset, gate = W.draw_layer_inputs(cfg)
    if gate_mode == "all":
        gate = np.ones(cfg.T, np.uint8)
    ref, gp = _make_layer(moet, cfg.H, cfg.I, cfg.E, dset, cfg=cfg)
    yg, err = _run_forward(moet, logits, xb, cfg.k, gp, cfg.E, cfg.H, dset, gate)
    assert err == 0
    yo = _oracle_forward(logits, xb, cfg.k, ref, dset, gate, cfg.E)
    check_y(yg, yo)


@pytest.mark.parametrize("T", [1, 9, 33, 100, 300, 512, 513, 600])
def test_forward_mid_size(moet, T):
    """Several row tiles, K chunks, N-tiles and work items (T=300 gives > 64 pairs per
    expert; T <= 512 runs the block-scaled decode engine, T > 512 the bf16 prefill engine)."""
    H, I, E, k = 1024, 256, 16, 4
    rng = np.random.default_rng(30 + T)
    dset = np.array([1, 4, 5, 11], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.5).astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))
    # no delta arguments at all
    yg2, _ = _run_forward(moet, logits, xb, k, gp, E, H)
    check_y(yg2, _oracle_forward(logits, xb, k, ref))


@pytest.mark.parametrize("T", [64, 600])
def test_forward_extreme_token_magnitudes(moet, T):
    """Tokens scaled by 1e-12 and 1e+12 and an all-zero token, each group held to the layer
    tolerance on its own (a global check would not see a tiny token): the activation scaling of
    both engines -- per-token NVFP4 term scales (T = 64) and the per-row power-of-two scaling of
    h into fp16 (T = 600) -- must follow the magnitude."""
    H, I, E, k = 1024, 256, 16, 4
    rng = np.random.default_rng(70 + T)
    dset = np.array([2, 7, 9], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, H)).astype(np.float32)
    tiny, huge, zero = np.arange(0, 5), np.arange(5, 10), 10
    x[tiny] *= np.float32(1e-12)
    x[huge] *= np.float32(1e12)
    x[zero] = 0.0
    xb = W.f32_to_bf16_bits(x)
    gate = (rng.random(T) < 0.5).astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    yo = _oracle_forward(logits, xb, k, ref, dset, gate, E)
    yg = np.asarray(yg, np.float64)
    for rows in (tiny, huge, np.arange(11, T)):
        check_y(yg[rows], yo[rows])
    assert not yg[zero].any() and not yo[zero].any()


@pytest.mark.parametrize("gate_mode", ["draw", "all", "none"])
def test_forward_prefill_ragged_items(moet, gate_mode):
    """Prefill engine with experts of more than 256 pairs: items split at 256 with a ragged
    tail (T=1100, E=8, k=2: about 275 pairs per expert), every token checked; the delta pass
    with some, all or no gated tokens."""
    H, I, E, k, T = 512, 256, 8, 2, 1100
    rng = np.random.default_rng(60)
    dset = np.array([0, 3, 6], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = {"draw": (rng.random(T) < 0.3), "all": np.ones(T, bool), "none": np.zeros(T, bool)}[gate_mode]
    gate = gate.astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


@pytest.mark.parametrize("I", [4352, 12288], ids=["two_per_thread", "four_per_thread"])
def test_forward_prefill_wide_intermediate(moet, I):
    """Prefill engine with an intermediate size whose h row spans more than 256 threads' output
    pairs (I / 16 = 272: two per thread, the last thread's second pair past the row; I / 16 = 768:
    four per thread; about 300 pairs per expert, so items split at 256): the h -> fp16 step holds a row of h in registers, takes its max |h| there and
    writes the permuted fp16 row and its gated copy from the same registers.  Every token checked."""
    H, E, k, T = 256, 4, 2, 600
    rng = np.random.default_rng(200 + I)
    dset = np.array([1, 3], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.3).astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


@pytest.mark.parametrize("gate_mode", ["draw", "all"])
def test_forward_prefill_two_lists(moet, gate_mode):
    """Prefill regime with skewed routing (a Zipf logit bias over 64 experts): hot experts (more
    than 64 pairs) run in the bf16 engine, the others in the block-scaled decode engine as a second
    work list with term rows per item slot; delta experts on both sides, every token checked."""
    H, I, E, k, T = 1024, 256, 64, 4, 700
    rng = np.random.default_rng(190)
    dset = np.array([0, 1, 5, 17, 40, 63], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    bias = np.log(np.arange(1, E + 1, dtype=np.float64) ** -1.1)[rng.permutation(E)]
    logits = (rng.standard_normal((T, E)) + bias).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = ((rng.random(T) < 0.3) if gate_mode == "draw" else np.ones(T, bool)).astype(np.uint8)
    counts = np.bincount(oroute.route_topk(logits, k)[0].ravel(), minlength=E)
    assert (counts > 64).sum() >= 4 and ((counts > 0) & (counts <= 64)).sum() >= 20
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


@pytest.mark.parametrize("T", [64, 700], ids=["decode_engine", "prefill_engines"])
def test_forward_pair_order_within_experts_leaves_y_unchanged(moet, T):
    """Any order of the pairs inside each expert's bucket gives the same y bit for bit: every
    pair's result depends only on its own column (the prefill regime relies on this when it
    walks each cached expert's gated pairs first).  Skewed routing over 64 experts with delta
    experts and a gate mask; the bucketing permutation is shuffled within every expert's range."""
    H, I, E, k = 1024, 256, 64, 4
    rng = np.random.default_rng(230 + T)
    dset = np.array([0, 1, 5, 17, 40, 63], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    bias = np.log(np.arange(1, E + 1, dtype=np.float64) ** -1.1)[rng.permutation(E)]
    logits = (rng.standard_normal((T, E)) + bias).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.3).astype(np.uint8)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(dev(logits), k, idx, w, off, perm)
    x = dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    dkw = dict(delta_slot=dev(W.delta_slot_table(E, dset)), dfc1=gp[1, "d"], dfc2=gp[2, "d"], gate_mask=dev(gate))
    ys = []
    offs, pm = off.cpu().numpy(), perm.cpu().numpy()
    for shuffle in (False, True):
        pr = pm.copy()
        if shuffle:
            for e in range(E):
                seg = pr[offs[e]:offs[e + 1]]
                pr[offs[e]:offs[e + 1]] = seg[rng.permutation(len(seg))]
            assert not np.array_equal(pr, pm)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        moet.moe_forward(x, idx, w, off, dev(pr), gp[1], gp[2], y, ws, **dkw)
        ys.append(y)
    torch.cuda.synchronize()
    assert moet.last_device_error() == 0
    assert torch.equal(ys[0], ys[1])


@pytest.mark.parametrize("T", [100, 700])
def test_forward_mma_sync_engine(moet, T):
    """Shapes the tcgen05 engines do not take (I = 384, not a multiple of 256) run the
    mma.sync engine at any token count."""
    H, I, E, k = 1024, 384, 16, 4
    rng = np.random.default_rng(70 + T)
    dset = np.array([2, 9], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.5).astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


def _pool_planes(moet, gp, experts):
    """Pool slots s = 0.. holding the planes of experts[s] (a gather of the full planes)."""
    ix = torch.tensor(np.asarray(experts, np.int64), device=DEV)
    return {f: moet.Planes(gp[f].sign.index_select(0, ix).contiguous(), gp[f].mag.index_select(0, ix).contiguous(),
                           gp[f].s16.index_select(0, ix).contiguous(), gp[f].scale_2.index_select(0, ix).contiguous())
            for f in (1, 2)}


@pytest.mark.parametrize("T,I", [(9, 256), (600, 256), (100, 384)])
def test_forward_pooled(moet, T, I):
    """Forward over a pool of resident experts (decode engine T=9, prefill engine T=600, mma.sync
    engine I=384): non-resident routed experts contribute zero and are counted exactly; with
    every expert resident, in any slot order, the result equals the full forward bit for bit
    (the fetch-and-replay of the README's expert cache)."""
    H, E, k = 1024, 16, 4
    rng = np.random.default_rng(90 + T + I)
    dset = np.array([1, 4, 5, 11], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.5).astype(np.uint8)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(dev(logits), k, idx, w, off, perm)
    x = dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    dkw = dict(delta_slot=dev(W.delta_slot_table(E, dset)), dfc1=gp[1, "d"], dfc2=gp[2, "d"], gate_mask=dev(gate))
    y_full = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moet.moe_forward(x, idx, w, off, perm, gp[1], gp[2], y_full, ws, **dkw)

    # 9 of 16 experts resident, in shuffled pool slots
    pool = rng.permutation(E)[:9]
    slot = np.full(E, -1, np.int32)
    slot[pool] = np.arange(len(pool), dtype=np.int32)
    pp = _pool_planes(moet, gp, pool)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    miss = torch.zeros(1, dtype=torch.int32, device=DEV)
    mask = torch.zeros(E, dtype=torch.uint8, device=DEV)
    moet.moe_forward_pooled(x, idx, w, off, perm, dev(slot), pp[1], pp[2], y, ws, miss_count=miss, miss_mask=mask,
                            **dkw)
    assert moet.last_device_error() == 0
    idx_np = idx.cpu().numpy()
    resident = slot >= 0
    assert int(miss.item()) == int(np.sum(~resident[idx_np]))
    routed = np.zeros(E, bool)
    routed[idx_np.ravel()] = True
    assert np.array_equal(mask.cpu().numpy().astype(bool), routed & ~resident)
    oi, ow = oroute.route_topk(logits, k)
    yo = omoe.moe_forward(W.bf16_bits_to_f32(xb).astype(np.float64), oi, ow, ref[1], ref[2],
                          W.delta_slot_table(E, dset), ref[1, "d"], ref[2, "d"], gate, resident=resident)
    check_y(y.float().cpu().numpy(), yo)

    # fetch every expert into a pool of E slots in another order and replay: bit-identical
    order = rng.permutation(E)
    slot2 = np.empty(E, np.int32)
    slot2[order] = np.arange(E, dtype=np.int32)
    pp2 = _pool_planes(moet, gp, order)
    y2 = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    miss.zero_()
    moet.moe_forward_pooled(x, idx, w, off, perm, dev(slot2), pp2[1], pp2[2], y2, ws, miss_count=miss, **dkw)
    assert int(miss.item()) == 0
    assert torch.equal(y2, y_full)


def test_forward_pooled_slot_out_of_range_sets_device_flag(moet):
    H, I, E, k, T = 256, 128, 8, 2, 8
    rng = np.random.default_rng(42)
    _, gp = _make_layer(moet, H, I, E, np.array([0], np.int32), rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(dev(logits), k, idx, w, off, perm)
    x = dev(W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).view(np.int16)).view(torch.bfloat16)
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    pp = _pool_planes(moet, gp, np.arange(4))
    slot = np.array([0, 1, 2, 3, 9, 9, 9, 9], np.int32)       # slots 9 do not exist in a pool of 4
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moet.moe_forward_pooled(x, idx, w, off, perm, dev(slot), pp[1], pp[2], y, ws)
    assert moet.last_device_error() == 8                        # MOET_ERR_DEVICE_INDEX
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (64, 256, 8), (300, 16, 4)])
def test_gate_from_confidence_bit_exact(moet, T, E, k):
    rng = np.random.default_rng(100 + T)
    conf = rng.random(T).astype(np.float32)
    conf[::7] = np.float32(0.6)                              # exactly tau: not gated
    conf[1::11] = np.nan
    conf[2::13] = -np.inf
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    slot = np.full(E, -1, np.int32)
    cached = rng.permutation(E)[: E // 3]
    slot[cached] = np.arange(len(cached), dtype=np.int32)
    gate = torch.zeros(T, dtype=torch.uint8, device=DEV)
    need = torch.zeros(E, dtype=torch.uint8, device=DEV)
    counts = torch.zeros(2, dtype=torch.int32, device=DEV)
    moet.gate_from_confidence(dev(conf), 0.6, dev(idx), gate, delta_slot=dev(slot), need_mask=need, counts=counts)
    assert moet.last_device_error() == 0
    g, nd, ng, npairs = ogate.gate_from_confidence(conf, 0.6, idx, slot)
    assert np.array_equal(host(gate), g)
    assert np.array_equal(host(need).astype(bool), nd)
    assert host(counts).tolist() == [ng, npairs]


def test_gate_replay_promotes_and_decides_again(moet):
    """The gate's replay: gate from confidence, promote every expert it asks for into the delta
    cache (their delta codes are already in the pool; the slot table is updated), replay the
    forward; the result equals the oracle with those slots, and a second decision asks for
    nothing."""
    H, I, E, k, T = 1024, 256, 16, 4, 33
    rng = np.random.default_rng(110)
    # every expert's delta in pool slot e; at first only a few experts hold a slot
    ref, gp = _make_layer(moet, H, I, E, np.arange(E, dtype=np.int32), rng=rng)
    slot = np.full(E, -1, np.int32)
    slot[[2, 7, 11]] = [2, 7, 11]
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    conf = rng.random(T).astype(np.float32)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    moet.route_topk(dev(logits), k, idx, w, off, perm)
    gate = torch.zeros(T, dtype=torch.uint8, device=DEV)
    need = torch.zeros(E, dtype=torch.uint8, device=DEV)
    counts = torch.zeros(2, dtype=torch.int32, device=DEV)
    moet.gate_from_confidence(dev(conf), 0.6, idx, gate, delta_slot=dev(slot), need_mask=need, counts=counts)
    # the oracle decides on its own routing; the GPU's decision must match it bit for bit
    oi, _ = oroute.route_topk(logits, k)
    gate_o, need_o, _, npairs_o = ogate.gate_from_confidence(conf, 0.6, oi, slot)
    assert np.array_equal(host(gate), gate_o) and np.array_equal(host(need).astype(bool), need_o)
    assert need_o.any() and host(counts)[1] == npairs_o
    slot2 = slot.copy()
    slot2[need_o] = np.flatnonzero(need_o).astype(np.int32)            # promote
    x = dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moet.moe_forward(x, idx, w, off, perm, gp[1], gp[2], y, ws, delta_slot=dev(slot2), dfc1=gp[1, "d"],
                     dfc2=gp[2, "d"], gate_mask=gate)
    assert moet.last_device_error() == 0
    yo = _oracle_forward(logits, xb, k, ref, np.arange(E, dtype=np.int32), gate_o, E, slot=slot2)
    check_y(y.float().cpu().numpy(), yo)
    # decide again with the promoted table: nothing left to promote
    need.zero_(); counts.zero_()
    moet.gate_from_confidence(dev(conf), 0.6, idx, gate, delta_slot=dev(slot2), need_mask=need, counts=counts)
    assert not host(need).any() and host(counts)[1] == 0


@pytest.mark.parametrize("T", [300, 600])
def test_forward_all_tokens_on_the_same_experts(moet, T):
    """Degenerate routing: every token picks the same k experts (a logit bias), so each of them
    gets T pairs split into many work items with a ragged last one (16-pair items in the decode
    engine at T=300, 256-pair items in the prefill engine at T=600); the other experts get none."""
    H, I, E, k = 512, 256, 16, 4
    rng = np.random.default_rng(120 + T)
    dset = np.array([3, 9], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, [3, 5, 9, 12]] += 50.0
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.4).astype(np.uint8)
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


def test_forward_max_experts_and_k(moet):
    """E = 1024 experts and k = 16 (the interface's maxima) on random planes: most routed experts
    get a single pair, each token sums 16 pairs."""
    H, I, E, k, T = 256, 256, 1024, 16, 5
    rng = np.random.default_rng(130)
    ref, gp = {}, {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        pl = _random_planes(rng, E, N, K)
        ref[f] = pl
        gp[f] = moet.Planes(dev(pl["sign"].view(np.int32)), dev(pl["mag"].view(np.int32)), dev(pl["s16"]),
                            dev(pl["scale_2"]))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref))


def test_forward_is_deterministic(moet):
    H, I, E, k, T = 1024, 256, 16, 4, 100
    rng = np.random.default_rng(40)
    dset = np.array([0, 2], dtype=np.int32)
    _, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = np.ones(T, np.uint8)
    a, _ = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    b, _ = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert np.array_equal(a, b)


def test_forward_bad_slot_sets_device_flag(moet):
    H, I, E, k, T = 256, 128, 8, 2, 8
    rng = np.random.default_rng(41)
    dset = np.array([0, 1], dtype=np.int32)
    _, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    slot = np.full(E, 7, np.int32)                 # pool has 2 slots
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, np.ones(T, np.uint8), slot=slot)
    assert err == 8                                # MOET_ERR_DEVICE_INDEX
    assert np.all(np.isfinite(yg))
    assert moet.last_device_error() == 0           # cleared by the read


@pytest.mark.parametrize("T", [9, 600], ids=["decode_engine", "prefill_engine"])
def test_bounded_wait_expiry_reports_timeout_and_recovers(moet, T):
    """A wait that runs out: with the poll bound lowered and CTA 0 of each engine launch withholding
    its first unit record (moet_debug_wait_expiry), every role waiting on that record gives up,
    the CTA releases TMEM and leaves, and the forward reports MOET_ERR_TIMEOUT without faulting.
    Afterwards, with the defaults restored, the same forward completes and matches the oracle (the
    context is intact, no TMEM was left allocated, no copy left in flight)."""
    H, I, E, k = 1024, 256, 16, 4
    rng = np.random.default_rng(180 + T)
    dset = np.array([3, 8], dtype=np.int32)
    ref, gp = _make_layer(moet, H, I, E, dset, rng=rng)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    gate = (rng.random(T) < 0.5).astype(np.uint8)
    assert moet.last_device_error() == 0
    moet.debug_wait_expiry(20000, True)
    try:
        _, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    finally:
        moet.debug_wait_expiry()
    assert moet.status_string(err) == "MOET_ERR_TIMEOUT"
    assert moet.last_device_error() == 0                    # read and cleared
    yg, err = _run_forward(moet, logits, xb, k, gp, E, H, dset, gate)
    assert err == 0
    check_y(yg, _oracle_forward(logits, xb, k, ref, dset, gate, E))


# ------------------------------------------------------------------ full-size layers, sampled tokens
def _random_planes(rng, E, N, K):
    sign = rng.integers(0, 2 ** 32, (E, N, K // 32), dtype=np.uint32)
    mag = rng.integers(0, 2 ** 32, (E, N, K // 32), dtype=np.uint32)
    s16 = rng.integers(40, 57, (E, N, K // 16), dtype=np.uint8)
    sc2 = (rng.random(E) * 0.004 + 0.004).astype(np.float32)
    return dict(sign=sign, mag=mag, s16=s16, scale_2=sc2)


# Full-size layers: the planes of every expert come from the seeded generators in `workloads`
# (drawn on the host, one (expert, FC) matrix at a time, and uploaded); the oracle regenerates
# the planes of the experts the sampled tokens route to, in spawn-started worker processes
# (`_oracle_shard`), one shard of experts each.
FULL_SEED = 50
FULL_CASES = {
    # name: (config, sampled tokens or a rule, gate override)
    "dsv3_decode_t1": ("dsv3_decode_t1", "all", None),
    "dsv3_decode_t1_gated": ("dsv3_decode_t1", "all", "all"),
    "dsv3_decode_t8": ("dsv3_decode_t8", "all", None),
    "dsv3_decode_t64": ("dsv3_decode_t64", "mix", None),
    "glm_decode": ("glm_decode", "all", None),
    "kimi_layer": ("kimi_layer", "spread", None),
    "dsv3_prefill": ("dsv3_prefill", "mix", None),
}


def _full_layer_gpu(moet, cfg, n_slots):
    """GPU planes [E, ...] and delta pool [n_slots, ...] drawn by the shared generators."""
    heavy = cfg.dist == "student_t4"
    gp = {}
    for f, (N, K) in ((1, (2 * cfg.I, cfg.H)), (2, (cfg.H, cfg.I))):
        sign = torch.empty((cfg.E, N, K // 32), dtype=torch.int32, device=DEV)
        mag = torch.empty_like(sign)
        s16 = torch.empty((cfg.E, N, K // 16), dtype=torch.uint8, device=DEV)
        for e in range(cfg.E):
            sg, mg, sc = W.draw_plane_matrix(FULL_SEED, e, f, N, K, heavy)
            sign[e].copy_(torch.from_numpy(sg.view(np.int32)))
            mag[e].copy_(torch.from_numpy(mg.view(np.int32)))
            s16[e].copy_(torch.from_numpy(sc))
        gp[f] = moet.Planes(sign, mag, s16, dev(W.draw_plane_scale2(FULL_SEED, f, cfg.E, K)))
        S = max(n_slots, 1)
        codes = torch.zeros((S, N, K // 2), dtype=torch.uint8, device=DEV)
        s4 = torch.zeros((S, N, K // 16), dtype=torch.uint8, device=DEV)
        for s_ in range(n_slots):
            dc, ds = W.draw_delta_matrix(FULL_SEED, s_, f, N, K)
            codes[s_].copy_(torch.from_numpy(dc))
            s4[s_].copy_(torch.from_numpy(ds))
        gp[f, "d"] = moet.DeltaPool(codes, s4)
    return gp


def _sample_tokens(rule, T, gate):
    if rule == "all":
        return list(range(T))
    if rule == "spread":
        return sorted({int(t) for t in np.linspace(0, T - 1, 8).round()})
    # "mix": four gated and four ungated tokens (as many as the batch has)
    g = [int(t) for t in np.flatnonzero(gate != 0)]
    u = [int(t) for t in np.flatnonzero(gate == 0)]
    pick = g[:: max(1, len(g) // 4)][:4] + u[:: max(1, len(u) // 4)][:4]
    return sorted(set(pick))


def _oracle_full(cfg, logits, xb, gate, slot, tokens):
    """Oracle y for the sampled tokens, the experts split over spawn workers."""
    import multiprocessing as mp
    import os
    import _oracle_shard
    oi, ow = oroute.route_topk(logits, cfg.k)
    x = W.bf16_bits_to_f32(xb[tokens]).astype(np.float64)
    idx, wts = oi[tokens], ow[tokens]
    g = gate[tokens] if slot is not None else None
    experts = np.unique(idx)
    n = max(1, min(8, os.cpu_count() or 1, len(experts)))
    shards = [sh for sh in np.array_split(experts, n) if len(sh)]
    jobs = [(FULL_SEED, cfg.H, cfg.I, cfg.E, cfg.dist == "student_t4", x, idx, wts, g, slot, sh) for sh in shards]
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        parts = pool.map(_oracle_shard.shard_forward, jobs)
    return np.sum(parts, axis=0)


@pytest.mark.parametrize("case", list(FULL_CASES))
def test_forward_full_size_sampled(moet, case):
    """Every layer configuration at full size, the whole batch through the library, sampled
    tokens against the oracle: all tokens at T = 1 and 8 (GLM: every token gated), four gated and
    four ungated tokens at T = 64 and in the prefill batch, eight tokens spread over the 1T-class
    layer's 256.  Planes with block scales over the whole e4m3 range (subnormal and zero blocks
    included), wider still for the Student-t layers."""
    cname, rule, gate_override = FULL_CASES[case]
    cfg = W.CONFIGS[cname]
    logits, xb, dset, gate = W.draw_layer_inputs(cfg)
    if gate_override == "all":
        gate = np.ones(cfg.T, np.uint8)
    with_delta = len(dset) > 0 and cfg.gate != "none"
    gp = _full_layer_gpu(moet, cfg, len(dset) if with_delta else 0)
    yg, err = _run_forward(moet, logits, xb, cfg.k, gp, cfg.E, cfg.H, dset if with_delta else None, gate)
    assert err == 0
    assert np.all(np.isfinite(yg))
    tokens = _sample_tokens(rule, cfg.T, gate)
    slot = W.delta_slot_table(cfg.E, dset) if with_delta else None
    yo = _oracle_full(cfg, logits, xb, gate, slot, tokens)
    check_y(yg[tokens], yo, label=f"full-size {case} tokens={len(tokens)}")
    del gp
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- sign-bias probe
PROBE_CODEBOOKS = [(-2, -1, 0, 1), (-3, -1, 1, 3), (-4, -1, 1, 4)]


def _gpu_probe(moet, w, levels):
    M, N, K = w.shape
    rows = torch.empty((M, N, 4), dtype=torch.float64, device=DEV)
    sums = torch.empty((M, 4), dtype=torch.float64, device=DEV)
    moet.sign_bias_probe(dev(w), levels, rows, sums)
    torch.cuda.synchronize()
    return host(rows), host(sums)


def _check_probe_rows(got_rows, w, levels):
    """The kernel ranks the 969 candidates in fp32; the oracle decides exactly.  A block whose
    exact decision margin (relative gap from the best score to the next candidate's) exceeds the
    kernel's fp32 ranking error must get the exact choice: every row made only of such blocks
    equals the oracle's sums (fp64 summation order aside).  In a row with a closer block the
    kernel may take a candidate whose score is within that error, so its error sum may differ by
    at most that much of the block's score, and its bias is not compared.  Returns the number of
    rows held to the exact choice."""
    from oracle import signbias as osb
    per_block, margin, nbest, sabs = osb.probe_blocks(w, levels)
    ref = per_block.sum(axis=1)
    u = 2.0 ** -24
    # fp32 ranking error: N = A P[c1] + B P[c2] + C P[c3] + L3 P[16] from fp32 prefix sums (each
    # within 16 u sum|w| of exact), squared and cross-multiplied (a few u more)
    L0, L1, L2, L3 = levels
    coef = abs(L0 - L1) + abs(L1 - L2) + abs(L2 - L3) + abs(L3)
    with np.errstate(divide="ignore", invalid="ignore"):
        eps = np.where(nbest > 0, 2.0 * coef * 16 * u * sabs / nbest, 1.0) + 8 * u
    close = margin <= eps
    score = per_block[..., 1] - per_block[..., 3]            # Nc^2 / Dc of the exact choice
    scale = np.abs(ref).max()
    exact_rows = ~close.any(axis=1)
    assert np.allclose(got_rows[exact_rows], ref[exact_rows], rtol=1e-12, atol=1e-13 * scale)
    assert np.allclose(got_rows[:, :2], ref[:, :2], rtol=1e-12, atol=1e-13 * scale)
    tol = ((2 * eps + margin) * score * close).sum(axis=1) + 1e-12 * np.abs(ref[:, 3]) + 1e-13 * scale
    assert (np.abs(got_rows[:, 3] - ref[:, 3]) <= tol).all()
    return int(exact_rows.sum())


@pytest.mark.parametrize("levels", PROBE_CODEBOOKS)
def test_sign_bias_probe_matches_oracle(moet, levels):
    """Per-row and per-matrix sums against the exact oracle: ragged rows (33 blocks, so lanes hold
    unequal counts), zero blocks, one-signed blocks, repeated values and exact grid fits."""
    M, N, K = 3, 37, 528
    rng = np.random.default_rng(160)
    w = (rng.standard_t(4, (M, N, K)) * 0.02).astype(np.float32)
    w[0, 0, :16] = 0
    w[0, 1, :16] = np.abs(w[0, 1, :16])
    w[0, 2, 16:32] = -np.abs(w[0, 2, 16:32])
    w[1, 3, :16] = 0.01
    w[1, 4, :16] = np.float32(0.25) * np.asarray(levels, np.float32)[np.arange(16) % 4]
    w[2] *= np.float32(1e-3)
    rows, sums = _gpu_probe(moet, w, levels)
    held = 0
    for m in range(M):
        held += _check_probe_rows(rows[m], w[m], levels)
        assert np.array_equal(sums[m], np.cumsum(rows[m], axis=0)[-1])       # rows summed in order
    assert held >= 0.5 * M * N                  # most rows are held to the exact choice


def test_sign_bias_probe_full_size_sampled_rows(moet):
    """DeepSeek-V3 FC1-sized matrices [4096, 7168]: sampled rows against the exact oracle; the
    naive codebook's bias is negative on every matrix and the symmetric codebook's far smaller."""
    from oracle import signbias as osb
    rng = np.random.default_rng(161)
    M, N, K = 2, 4096, 7168
    w = (rng.standard_t(4, (M, N, K)) * (0.02 / np.sqrt(2))).astype(np.float32)
    stats = {}
    for levels in ((-2, -1, 0, 1), (-3, -1, 1, 3)):
        rows, sums = _gpu_probe(moet, w, levels)
        for m in range(M):
            sel = np.unique(np.r_[0, N - 1, rng.integers(0, N, 6)])
            _check_probe_rows(rows[m, sel], w[m, sel], levels)
        stats[levels] = [osb.statistics(sums[m], N * K) for m in range(M)]
    assert all(s["bias"] < -0.01 for s in stats[(-2, -1, 0, 1)])
    for a, b in zip(stats[(-3, -1, 1, 3)], stats[(-2, -1, 0, 1)]):
        assert abs(a["bias"]) * 10 < abs(b["bias"])


def test_sign_bias_probe_rejects_bad_levels(moet):
    w = torch.zeros((1, 2, 32), dtype=torch.float32, device=DEV)
    rows = torch.empty((1, 2, 4), dtype=torch.float64, device=DEV)
    sums = torch.empty((1, 4), dtype=torch.float64, device=DEV)
    for bad in ((-1, -1, 0, 1), (3, 1, -1, -3), (-100, -1, 1, 100)):
        with pytest.raises(moet.MoetError):
            moet.sign_bias_probe(w, bad, rows, sums)
