#!/usr/bin/env python
"""MoE-layer throughput of the 2-bit expert layer on one GB300 (or N replicas).

One step = the whole hot path on one batch: router top-k + bucketing
(moet_route_topk) and the MoE forward (moet_moe_forward: FC1 gate|up with
SiLU*mul, FC2 with the weighted combine, the NVFP4 delta on gated tokens of
cached experts) for the DeepSeek-V3-class decode layer (H=7168, I=2048,
E=256, k=8), T=64 tokens by default.  Inputs are resident in HBM; a step's
library calls are captured once into a CUDA graph and replayed; the L2 is
flushed (512 MB memset) before every step and each step is timed alone with
CUDA events on the launching stream.  Per-kernel durations (the roofline) come
from the same steps launched call by call with the library's event profiler.
The end-to-end number replays a graph of the step plus the host copies of its
inputs (pinned) and its output.  Every layer configuration (T=1 / 8 / 64,
prefill, GLM worst case, 1T-class) gets a compact record under "configs" at the
end of the line: tokens/s of the step and end to end, FC1 / FC2 time per step
and the roofline fractions.  The load-time requantisation is timed over the
full NVFP4 expert set of the 1T-class layer (768 matrices), planes only and
with the delta ("requant").  Other extras: the forward through the expert-cache
slot table ("pooled"), the FP8 and MXFP4 requantisations and the sign-bias
probe over 16 FC1-shaped matrices ("requant_fp8", "requant_mxfp4",
"sign_bias"); --extras picks a subset and --requant-experts shrinks the
requant set (profiler captures).

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300; weight-stream GB/s as % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_MIN_T = 512          # the library runs its bf16 prefill engine above this many tokens
L2_FLUSH_BYTES = 512 << 20
EXTRAS = ("sweep", "pooled", "requant", "requant_fp8", "requant_mxfp4", "sign_bias")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3_decode_t64")
    ap.add_argument("--no-extras", action="store_true", help="skip the T-sweep and the requant timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller layer for profiler captures; not a bench line)")
    ap.add_argument("--extras", default=",".join(EXTRAS),
                    help="comma list of the extra measurements to run (default: all of " + ",".join(EXTRAS) + ")")
    ap.add_argument("--requant-experts", type=int, default=0,
                    help="requant over this many experts of the 1T-class layer instead of all (profiler captures)")
    args = ap.parse_args()
    args.extras = {e for e in args.extras.split(",") if e}
    unknown = args.extras - set(EXTRAS)
    if unknown:
        ap.error(f"unknown extras {sorted(unknown)}")
    return args


def workload(args):
    import dataclasses
    cfg = W.CONFIGS[args.workload]
    if args.experts:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_e{args.experts}", E=args.experts,
                                  n_delta=min(cfg.n_delta, args.experts // 2))
    return cfg


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ peaks, clocks
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
                if key in d:
                    return float(d[key]), "measured"
            for key, v in d.items():
                if "hbm" in key.lower() and isinstance(v, (int, float)):
                    return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def fc1_traffic(workload):
    """FC1 DRAM bytes per launch from the committed ncu summary, or None when the summary was
    taken on another workload or another FC kernel source (the counters no longer apply)."""
    p = os.path.join(ROOT, "profiles", "fc1_traffic.txt")
    src = os.path.join(ROOT, "bit_moe_expert_moet_gb300", "csrc", "moe_tc.cu")
    if workload != "dsv3_decode_t64" or not (os.path.exists(p) and os.path.exists(src)):
        return None
    import hashlib
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    rec = {}
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 2 and not line.startswith("#"):
                rec[parts[0]] = parts[1]
    if rec.get("source_sha256") != sha:
        return None
    return int(rec["fc1_traffic_bytes"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 7:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": num(rows[0][1]),
                "power_w_median": statistics.median([num(r[2]) for r in rows]),
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ layer construction (GPU)
def gen_weight_chunk(torch, gen, dist_name, shape, dev):
    if dist_name == "normal":
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * 0.02
    z = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
    c = torch.zeros(shape, device=dev, dtype=torch.float32)
    for _ in range(4):
        c.add_(torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).square_())
    return z * torch.rsqrt(c * 0.25) * (0.02 / math.sqrt(2.0))


def build_layer(moet, torch, cfg, dset, dev, seed=0, chunk=16):
    """fp32 weights drawn on the GPU -> NVFP4 (library) -> 2-bit planes (+ delta pool)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + seed)
    E, H, I = cfg.E, cfg.H, cfg.I
    planes, pools = {}, {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        sign = torch.empty((E, N, K // 32), dtype=torch.int32, device=dev)
        mag = torch.empty_like(sign)
        s16 = torch.empty((E, N, K // 16), dtype=torch.uint8, device=dev)
        sc2 = torch.empty(E, dtype=torch.float32, device=dev)
        S = max(len(dset), 1)
        dcodes = torch.zeros((S, N, K // 2), dtype=torch.uint8, device=dev)
        ds4 = torch.zeros((S, N, K // 16), dtype=torch.uint8, device=dev)
        slot_of = {int(e): i for i, e in enumerate(dset)}
        codes = torch.empty((chunk, N, K // 2), dtype=torch.uint8, device=dev)
        s4 = torch.empty((chunk, N, K // 16), dtype=torch.uint8, device=dev)
        dc_tmp = torch.empty_like(codes)
        ds_tmp = torch.empty_like(s4)
        for e0 in range(0, E, chunk):
            m = min(chunk, E - e0)
            w = gen_weight_chunk(torch, gen, cfg.dist, (m, N, K), dev)
            moet.quantize_nvfp4(w, codes[:m], s4[:m], sc2[e0:e0 + m])
            del w
            moet.requant_2bit(codes[:m], s4[:m], sign[e0:e0 + m], mag[e0:e0 + m], s16[e0:e0 + m],
                              dc_tmp[:m], ds_tmp[:m])
            for e in range(e0, e0 + m):
                if e in slot_of:
                    dcodes[slot_of[e]].copy_(dc_tmp[e - e0])
                    ds4[slot_of[e]].copy_(ds_tmp[e - e0])
        planes[f] = moet.Planes(sign, mag, s16, sc2)
        pools[f] = moet.DeltaPool(dcodes, ds4)
        del codes, s4, dc_tmp, ds_tmp
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return planes, pools


def step_bytes(cfg, idx, gate, slot):
    """Algorithmic HBM bytes of one step and of the FC1 launch, from the actual routing."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    used = np.unique(idx)
    delta_used = set()
    for t in range(T):
        if gate[t]:
            for e in idx[t]:
                if slot[e] >= 0:
                    delta_used.add(int(e))
    We = 3 * H * I
    w1 = 2 * I * H
    total = len(used) * We * (2 / 8 + 1 / 16) + len(delta_used) * We * (4 / 8 + 1 / 16) \
        + 8 * len(used) + 2 * T * H + 2 * T * H + 4 * T * E
    fc1 = len(used) * w1 * (2 / 8 + 1 / 16) + len(delta_used) * w1 * (4 / 8 + 1 / 16) \
        + 4 * len(used) + 2 * T * H + 4 * T * k * I
    w2 = H * I
    fc2 = len(used) * w2 * (2 / 8 + 1 / 16) + len(delta_used) * w2 * (4 / 8 + 1 / 16) \
        + 4 * len(used) + 4 * T * k * I + 4 * T * k * H
    return total, fc1, fc2, len(used), len(delta_used)


def fc_flops(cfg, idx, gate, slot):
    """Algorithmic FLOPs of FC1 and FC2: 2 (2I) H and 2 H I per routed pair, again for every pair
    whose token is gated and whose expert has a cached delta (the delta pass)."""
    pairs = cfg.T * cfg.k
    dpairs = sum(1 for t in range(cfg.T) if gate[t] for e in idx[t] if slot[e] >= 0)
    return 2.0 * (2 * cfg.I) * cfg.H * (pairs + dpairs), 2.0 * cfg.H * cfg.I * (pairs + dpairs)


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            if "bf16_tflops" in d:
                return float(d["bf16_tflops"]), "measured (burst)"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def _r(v, sig=4):
    """v rounded to `sig` significant digits (keeps the one-line record short)."""
    if v is None or not isinstance(v, (int, float)) or v == 0 or not math.isfinite(v):
        return v
    return float(f"{v:.{sig}g}")


def config_summary(l, step_ms, e2e_ms, prof, nsteps, peak):
    """Compact record of one layer configuration: tokens/s of the graph-replayed step and of the
    end-to-end step (host copies inside), per-step FC1 / FC2 kernel time from the event profiler
    (all launches of a kind in a step summed), and the roofline fractions: HBM (algorithmic bytes
    over the copy peak) for decode, bf16 tensor (useful FLOPs over the bf16 peak) for prefill."""
    c = l.cfg
    f1 = prof["fc1"][2] / nsteps
    f2 = prof["fc2"][2] / nsteps
    out = {"T": c.T, "tok_s": _r(c.T / (step_ms * 1e-3)), "e2e_tok_s": _r(c.T / (e2e_ms * 1e-3)),
           "step_ms": _r(step_ms), "fc1_ms": _r(f1), "fc2_ms": _r(f2)}
    if c.T > PREFILL_MIN_T:
        tpk, _ = bf16_peak()
        tf = 6.0 * c.H * c.I * c.T * c.k / (step_ms * 1e-3) / 1e12
        out.update({"tflops": _r(tf), "frac_bf16": _r(tf / tpk),
                    "fc1_frac_bf16": _r(l.flops_fc1 / (f1 * 1e-3) / 1e12 / tpk),
                    "fc2_frac_bf16": _r(l.flops_fc2 / (f2 * 1e-3) / 1e12 / tpk)})
    else:
        out.update({"step_frac_hbm": _r(l.bytes_total / (step_ms * 1e-3) / 1e9 / peak),
                    "fc1_frac_hbm": _r(l.bytes_fc1 / (f1 * 1e-3) / 1e9 / peak),
                    "fc2_frac_hbm": _r(l.bytes_fc2 / (f2 * 1e-3) / 1e9 / peak)})
    return out


class Layer:
    """One MoE layer resident on the GPU plus one batch of inputs."""

    def __init__(self, moet, torch, cfg, dev, seed=0, planes=None, pools=None, slot_np=None):
        self.moet, self.torch, self.cfg, self.dev = moet, torch, cfg, dev
        logits, xb, dset, gate = W.draw_layer_inputs(cfg)
        if planes is None:
            self.slot_np = W.delta_slot_table(cfg.E, dset)
            self.planes, self.pools = build_layer(moet, torch, cfg, dset, dev, seed=seed)
            self.n_slots_cfg = len(dset)
        else:
            self.slot_np, self.planes, self.pools = slot_np, planes, pools
            self.n_slots_cfg = int((slot_np >= 0).sum())
        self._set_batch(logits, xb, gate)

    def rebatch(self, cfg2):
        """Same weights and delta cache, another batch (a config with the same layer shape)."""
        return Layer(self.moet, self.torch, cfg2, self.dev, planes=self.planes, pools=self.pools,
                     slot_np=self.slot_np)

    def _set_batch(self, logits, xb, gate):
        t, cfg, dev, moet = self.torch, self.cfg, self.dev, self.moet
        T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
        self.gate_np = gate
        self.logits = t.from_numpy(logits).to(dev)
        self.x = t.from_numpy(xb.view(np.int16)).to(dev).view(t.bfloat16)
        self.gate = t.from_numpy(gate).to(dev)
        self.slot = t.from_numpy(self.slot_np).to(dev)
        self.idx = t.empty((T, k), dtype=t.int32, device=dev)
        self.w = t.empty((T, k), dtype=t.float32, device=dev)
        self.off = t.empty(E + 1, dtype=t.int32, device=dev)
        self.perm = t.empty(T * k, dtype=t.int32, device=dev)
        self.y = t.empty((T, H), dtype=t.bfloat16, device=dev)
        self.ws = t.empty(moet.forward_workspace_size(T, H, I, E, k), dtype=t.uint8, device=dev)
        self.use_delta = self.n_slots_cfg > 0 and cfg.gate != "none"
        # host-side buffers of the end-to-end path (pinned)
        self.h_logits = t.from_numpy(logits).pin_memory()
        self.h_x = t.from_numpy(xb.view(np.int16)).pin_memory()
        self.h_y = t.empty((T, H), dtype=t.int16).pin_memory()
        self.step()
        t.cuda.synchronize(dev)
        self.idx_np = self.idx.cpu().numpy()
        self.bytes_total, self.bytes_fc1, self.bytes_fc2, self.n_used, self.n_delta = step_bytes(
            cfg, self.idx_np, gate, self.slot_np)
        gate_eff = gate if self.use_delta else np.zeros_like(gate)
        self.flops_fc1, self.flops_fc2 = fc_flops(cfg, self.idx_np, gate_eff, self.slot_np)

    def step(self):
        m = self.moet
        m.route_topk(self.logits, self.cfg.k, self.idx, self.w, self.off, self.perm)
        kw = {}
        if self.use_delta:
            kw = dict(delta_slot=self.slot, dfc1=self.pools[1], dfc2=self.pools[2], gate_mask=self.gate)
        m.moe_forward(self.x, self.idx, self.w, self.off, self.perm, self.planes[1], self.planes[2],
                      self.y, self.ws, **kw)

    def step_e2e(self):
        self.logits.copy_(self.h_logits, non_blocking=True)
        self.x.view(self.torch.int16).copy_(self.h_x, non_blocking=True)
        self.step()
        self.h_y.copy_(self.y.view(self.torch.int16), non_blocking=True)

    @property
    def h2d_bytes(self):
        return self.h_logits.numel() * 4 + self.h_x.numel() * 2

    @property
    def d2h_bytes(self):
        return self.h_y.numel() * 2


def time_steps(torch, fn, steps, warmup, flush):
    """Per-step CUDA-event times (ms), L2 flushed before each step (outside the events)."""
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.fill_(1)
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush.fill_(1)
        a.record(st)
        fn()
        b.record(st)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def capture_graph(torch, fn):
    """One CUDA graph of fn's launches (all library calls are graph-capturable: static
    buffers, no host synchronisation); warmed once on a side stream first."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_requant_fp8(moet, torch, dev, steps=3, n_mat=16):
    """moet_requant_fp8_2bit over n_mat FP8 block-quant matrices of the DeepSeek-V3 FC1 shape
    [2I, H] = [4096, 7168] (random codes, the NaN codes excluded; random 128x128 block scales),
    with the delta.  Per weight 1 B in, 0.3125 + 0.5625 B out."""
    N, K = 4096, 7168
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    codes = torch.randint(0, 256, (n_mat, N, K), dtype=torch.uint8, device=dev, generator=g)
    codes[(codes & 0x7F) == 0x7F] ^= 1
    bs = torch.rand((n_mat, N // 128, K // 128), device=dev, generator=g) * 0.02 + 0.001
    sc2 = torch.empty(n_mat, dtype=torch.float32, device=dev)
    sign = torch.empty((n_mat, N, K // 32), dtype=torch.int32, device=dev)
    mag = torch.empty_like(sign)
    s16 = torch.empty((n_mat, N, K // 16), dtype=torch.uint8, device=dev)
    dcodes = torch.empty((n_mat, N, K // 2), dtype=torch.uint8, device=dev)
    ds4 = torch.empty_like(s16)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def run():
        moet.requant_fp8_2bit(codes, bs, sc2, sign, mag, s16, dcodes, ds4)

    ts = time_steps(torch, run, steps, 1, flush)
    ms = statistics.median(ts)
    weights = n_mat * N * K
    moved = weights * (1 + 0.3125 + 0.5625)
    return {"matrices": n_mat, "ms": _r(ms), "gw_s": _r(weights / (ms * 1e-3) / 1e9),
            "gbs": _r(moved / (ms * 1e-3) / 1e9)}


def time_requant_mxfp4(moet, torch, dev, steps=3, n_mat=16):
    """moet_requant_mxfp4_2bit over n_mat MXFP4 matrices of the DeepSeek-V3 FC1 shape
    [2I, H] = [4096, 7168] (random codes, random E8M0 exponents 2^-10 .. 2^-4), with the delta.
    Per weight 0.5 + 1/32 B in, 0.3125 + 0.5625 B out."""
    N, K = 4096, 7168
    g = torch.Generator(device=dev)
    g.manual_seed(8)
    codes = torch.randint(0, 256, (n_mat, N, K // 2), dtype=torch.uint8, device=dev, generator=g)
    e8m0 = torch.randint(117, 124, (n_mat, N, K // 32), dtype=torch.uint8, device=dev, generator=g)
    sc2 = torch.empty(n_mat, dtype=torch.float32, device=dev)
    sign = torch.empty((n_mat, N, K // 32), dtype=torch.int32, device=dev)
    mag = torch.empty_like(sign)
    s16 = torch.empty((n_mat, N, K // 16), dtype=torch.uint8, device=dev)
    dcodes = torch.empty((n_mat, N, K // 2), dtype=torch.uint8, device=dev)
    ds4 = torch.empty_like(s16)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def run():
        moet.requant_mxfp4_2bit(codes, e8m0, sc2, sign, mag, s16, dcodes, ds4)

    ts = time_steps(torch, run, steps, 1, flush)
    ms = statistics.median(ts)
    weights = n_mat * N * K
    moved = weights * (0.5 + 1 / 32 + 0.3125 + 0.5625)
    return {"matrices": n_mat, "ms": _r(ms), "gw_s": _r(weights / (ms * 1e-3) / 1e9),
            "gbs": _r(moved / (ms * 1e-3) / 1e9)}


def time_sign_bias_probe(moet, torch, dev, steps=3, n_mat=16):
    """moet_sign_bias_probe over n_mat fp32 matrices of the DeepSeek-V3 FC1 shape [4096, 7168]
    (Student-t(4) weights, std 0.02) for the naive int2 codebook and the two symmetric ones: the
    time per pass and the per-matrix bias and rel-RMS (mean, and the share of negative biases)."""
    N, K = 4096, 7168
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    w = gen_weight_chunk(torch, g, "t4", (n_mat, N, K), dev)
    rows = torch.empty((n_mat, N, 4), dtype=torch.float64, device=dev)
    sums = torch.empty((n_mat, 4), dtype=torch.float64, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {"matrices": n_mat}
    for name, levels in (("int2", (-2, -1, 0, 1)), ("sym13", (-3, -1, 1, 3)), ("sym14", (-4, -1, 1, 4))):
        ts = time_steps(torch, lambda: moet.sign_bias_probe(w, levels, rows, sums), steps, 1, flush)
        s = sums.cpu().numpy()
        n = N * K
        rms = np.sqrt(s[:, 1] / n)
        bias = s[:, 2] / n / rms
        rel = np.sqrt(s[:, 3] / s[:, 1])
        out[name] = {"ms": _r(statistics.median(ts)), "bias": _r(float(bias.mean()), 3),
                     "neg": _r(float((bias < 0).mean()), 3), "rel_rms": _r(float(rel.mean()), 3)}
    out["int2_over_sym13"] = _r(abs(out["int2"]["bias"]) / max(abs(out["sym13"]["bias"]), 1e-300), 3)
    del w, rows, flush
    torch.cuda.empty_cache()
    return out


def time_requant(moet, torch, dev, peak, steps=3, n_experts=0):
    """moet_requant_2bit over the full NVFP4 expert set of the 1T-class layer (768 matrices, or the
    first n_experts experts' matrices): one pass writing the planes only, one pass writing the
    planes and the NVFP4 delta (what filling the delta cache costs).  Bytes moved per pass are the
    tensors read and written; the fraction is of the copy peak."""
    cfg = W.CONFIGS["kimi_layer"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(99)
    E, H, I = (n_experts or cfg.E), cfg.H, cfg.I
    bufs = {}
    for f, (N, K) in ((1, (2 * I, H)), (2, (H, I))):
        codes = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
        s4 = torch.empty((E, N, K // 16), dtype=torch.uint8, device=dev)
        sc2 = torch.empty(E, dtype=torch.float32, device=dev)
        for e0 in range(0, E, 16):
            e1 = min(E, e0 + 16)
            w = gen_weight_chunk(torch, gen, cfg.dist, (e1 - e0, N, K), dev)
            moet.quantize_nvfp4(w, codes[e0:e1], s4[e0:e1], sc2[e0:e1])
            del w
        sign = torch.empty((E, N, K // 32), dtype=torch.int32, device=dev)
        mag = torch.empty_like(sign)
        s16 = torch.empty((E, N, K // 16), dtype=torch.uint8, device=dev)
        dcodes = torch.empty_like(codes)
        ds4 = torch.empty_like(s4)
        bufs[f] = (codes, s4, sign, mag, s16, dcodes, ds4)
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {"matrices": 2 * E, "weights": 3 * H * I * E}
    for name, with_delta in (("planes", False), ("delta", True)):
        def run():
            for f in (1, 2):
                codes, s4, sign, mag, s16, dcodes, ds4 = bufs[f]
                if with_delta:
                    moet.requant_2bit(codes, s4, sign, mag, s16, dcodes, ds4)
                else:
                    moet.requant_2bit(codes, s4, sign, mag, s16)
        ts = time_steps(torch, run, steps, 1, flush)
        nbytes = sum(t.numel() * t.element_size() for f in (1, 2) for t in bufs[f][:5 + 2 * with_delta])
        ms = statistics.median(ts)
        out[name] = {"ms": _r(ms), "gbs": _r(nbytes / (ms * 1e-3) / 1e9), "frac_hbm": _r(nbytes / (ms * 1e-3) / 1e9 / peak),
                     "bytes": nbytes}
    del bufs, flush
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample(cfg, n_pairs=1, seed=7):
    """Time the oracle on a bounded sample: route all T tokens, then the forward
    of the first n_pairs (token, expert) pairs of token 0, on random 2-bit planes
    drawn on the host.  Returns (tokens processed, seconds, description)."""
    from oracle import moe as omoe, route as oroute
    logits, xb, dset, gate = W.draw_layer_inputs(cfg)
    rng = np.random.default_rng(seed)
    E, H, I, k = cfg.E, cfg.H, cfg.I, cfg.k
    oi, ow = oroute.route_topk(logits[:1], k)
    experts = [int(e) for e in oi[0, :n_pairs]]
    def planes(N, K):
        return dict(sign=np.zeros((E, N, K // 32), np.uint32), mag=np.zeros((E, N, K // 32), np.uint32),
                    s16=np.zeros((E, N, K // 16), np.uint8), scale_2=np.full(E, 0.005, np.float32))
    fc1, fc2 = planes(2 * I, H), planes(H, I)
    for e in experts:
        for p, (N, K) in ((fc1, (2 * I, H)), (fc2, (H, I))):
            p["sign"][e] = rng.integers(0, 2 ** 32, (N, K // 32), dtype=np.uint32)
            p["mag"][e] = rng.integers(0, 2 ** 32, (N, K // 32), dtype=np.uint32)
            p["s16"][e] = rng.integers(40, 57, (N, K // 16), dtype=np.uint8)
    x = W.bf16_bits_to_f32(xb[:1]).astype(np.float64)
    t0 = time.perf_counter()
    oroute.route_topk(logits, k)
    idx = oi[:, :n_pairs]
    wts = ow[:, :n_pairs]
    omoe.moe_forward(x, idx, wts, fc1, fc2)
    dt = time.perf_counter() - t0
    desc = f"route of all {cfg.T} tokens + forward of {n_pairs} (token, expert) pair = {n_pairs / k:.3f} token"
    return n_pairs / k, dt, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ main
def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = workload(args)
    for _ in range(args.warmup):
        oracle_sample(cfg)
    tok, sec = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        t, s, desc = oracle_sample(cfg)
        tok += t
        sec += s
    value = tok / sec
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    if rank == 0 or world == 1:
        g.build()
    barrier(world)
    import bit_moe_expert_moet_gb300 as moet

    cfg = workload(args)
    layer = Layer(moet, torch, cfg, dev, seed=rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak, peak_kind = hbm_peak()

    # a step is the library's route + forward calls replayed as one CUDA graph (the launch
    # sequence a serving loop would capture); e2e adds the host copies to the same graph
    step_graph = capture_graph(torch, layer.step)
    e2e_graph = capture_graph(torch, layer.step_e2e)

    # timed region: K steps, per-step events
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ts = time_steps(torch, step_graph.replay, args.steps, args.warmup, flush)
    barrier(world)
    total_ms = max_over_ranks(sum(ts), world)
    ms_step = total_ms / args.steps
    value = world * cfg.T * args.steps / (total_ms * 1e-3)

    # the same K steps launched one call at a time with the library's event profiler on:
    # per-launch kernel durations for the roofline and the launch count
    moet.profile_read()
    moet.profile_enable(True)
    time_steps(torch, layer.step, args.steps, args.warmup, flush)
    moet.profile_enable(False)
    prof = moet.profile_read()

    # e2e through host buffers
    ts_e2e = time_steps(torch, e2e_graph.replay, args.steps, args.warmup, flush)
    e2e_ms = max_over_ranks(sum(ts_e2e), world)
    e2e_value = world * cfg.T * args.steps / (e2e_ms * 1e-3)
    err = moet.last_device_error()

    fl, ft, fms = prof["fc1"]
    fc1_ms = fms / max(ft, 1)
    achieved = layer.bytes_fc1 / (fc1_ms * 1e-3) / 1e9
    total_launches = sum(v[0] for v in prof.values())
    launches_timed = total_launches * args.steps // (args.steps + args.warmup)

    extras = {}
    configs = {}
    if rank == 0:
        configs[cfg.name] = config_summary(layer, statistics.median(ts), statistics.median(ts_e2e), prof,
                                           args.steps + args.warmup, peak)
    if not args.no_extras and rank == 0:
        def timed(l2, steps, warmup):
            g2 = capture_graph(torch, l2.step)
            t2 = time_steps(torch, g2.replay, steps, warmup, flush)
            del g2
            g3 = capture_graph(torch, l2.step_e2e)
            t3 = time_steps(torch, g3.replay, steps, warmup, flush)
            del g3
            moet.profile_read()
            moet.profile_enable(True)
            time_steps(torch, l2.step, steps, warmup, flush)
            moet.profile_enable(False)
            p2 = moet.profile_read()
            return config_summary(l2, statistics.median(t2), statistics.median(t3), p2, steps + warmup, peak)

        for name in (("dsv3_decode_t1", "dsv3_decode_t8", "dsv3_prefill") if "sweep" in args.extras else ()):
            c2 = W.CONFIGS[name]
            if name == cfg.name or (c2.H, c2.I, c2.E) != (cfg.H, cfg.I, cfg.E):
                continue
            l2 = layer.rebatch(c2)
            configs[name] = timed(l2, args.steps if c2.T <= 512 else 5, args.warmup if c2.T <= 512 else 3)
            del l2
        for name in (("glm_decode", "kimi_layer") if "sweep" in args.extras else ()):
            if name == cfg.name:
                continue
            c3 = W.CONFIGS[name]
            l3 = Layer(moet, torch, c3, dev)
            configs[name] = timed(l3, args.steps, args.warmup)
            del l3
            torch.cuda.empty_cache()

        if "pooled" in args.extras:
            # expert cache: the headline layer through the slot table with every 10th expert not
            # resident (their pairs contribute zero and are counted); the planes stay where they are
            slot_np = np.arange(cfg.E, dtype=np.int32)
            slot_np[::10] = -1
            slot_t = torch.from_numpy(slot_np).to(dev)
            miss = torch.zeros(1, dtype=torch.int32, device=dev)
            kwp = {}
            if layer.use_delta:
                kwp = dict(delta_slot=layer.slot, dfc1=layer.pools[1], dfc2=layer.pools[2], gate_mask=layer.gate)

            def pooled_step():
                moet.route_topk(layer.logits, cfg.k, layer.idx, layer.w, layer.off, layer.perm)
                moet.moe_forward_pooled(layer.x, layer.idx, layer.w, layer.off, layer.perm, slot_t, layer.planes[1],
                                        layer.planes[2], layer.y, layer.ws, miss_count=miss, **kwp)

            gp_ = capture_graph(torch, pooled_step)
            miss.zero_()
            tp = time_steps(torch, gp_.replay, args.steps, args.warmup, flush)
            med = statistics.median(tp)
            n_replays = args.steps + args.warmup
            extras["pooled"] = {"resident": int((slot_np >= 0).sum()),
                                "missed_pairs": int(miss.item()) / n_replays,
                                "tok_s": _r(cfg.T / (med * 1e-3)), "step_ms": _r(med)}
            del gp_
        if "requant" in args.extras:
            extras["requant"] = time_requant(moet, torch, dev, peak, n_experts=args.requant_experts)
        if "requant_fp8" in args.extras:
            extras["requant_fp8"] = time_requant_fp8(moet, torch, dev)
        if "requant_mxfp4" in args.extras:
            extras["requant_mxfp4"] = time_requant_mxfp4(moet, torch, dev)
        if "sign_bias" in args.extras:
            extras["sign_bias"] = time_sign_bias_probe(moet, torch, dev)
    if configs:
        extras["configs"] = configs           # last: the most-read records sit at the end of the line

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, sec, desc = oracle_sample(cfg)
        cpu = {"value": tok / sec, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc}

    if rank != 0:
        return
    if cfg.T > PREFILL_MIN_T:
        # prefill regime: FC1 is a dense contraction on the tensor cores (useful FLOPs per step over
        # FC1's summed launch time in the step)
        tpk, tpk_kind = bf16_peak()
        f1_step = prof["fc1"][2] / (args.steps + args.warmup)
        tach = layer.flops_fc1 / (f1_step * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "FC1 (pf_fc_kernel<FC1> + fc_tc_kernel<FC1>)", "achieved": _r(tach),
                    "peak": tpk, "peak_source": tpk_kind, "unit": "TFLOP/s", "frac": _r(tach / tpk), "traffic": None,
                    "flops": layer.flops_fc1, "ms": _r(f1_step), "frac_fp8": _r(tach / (2.0 * tpk))}
        dtype = "bf16/fp16 tcgen05 on exact 2-bit weights (+ nvfp4 block-scaled for small items), fp32 acc"
    else:
        tr = fc1_traffic(cfg.name)
        roofline = {"bound": "hbm", "kernel": "fc_tc_kernel<FC1>", "achieved": _r(achieved), "peak": peak,
                    "peak_source": peak_kind, "unit": "GB/s", "frac": _r(achieved / peak), "traffic": tr,
                    "traffic_source": "profiles/fc1_traffic.txt (ncu, same kernel source sha256)" if tr else None,
                    "bytes": layer.bytes_fc1, "ms": _r(fc1_ms), "frac_8tbs": _r(achieved / 8000.0)}
        dtype = "nvfp4 block-scaled tcgen05 (2-bit levels as e2m1, activations as 4 nvfp4 terms), fp32 acc"
    if cpu is not None:
        cpu["value"] = _r(cpu["value"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype,
        "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k,
                   "delta_experts": int((layer.slot_np >= 0).sum()), "gate": cfg.gate,
                   "l2": "flushed before each step", "parallelism": f"replicas x{world}"},
        "step_frac_hbm": _r(layer.bytes_total / (ms_step * 1e-3) / 1e9 / peak),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": layer.h2d_bytes,
                "d2h_bytes_per_step": layer.d2h_bytes},
        "clocks": clk.summary(),
        "gpu_launches": launches_timed,
        "device_error": err,
    }
    line.update(extras)            # per-config records ("configs") come last
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
