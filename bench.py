#!/usr/bin/env python
"""Benchmark of the fused-chain hot path on GB300.

One step runs every fused workload once, at full size, through the C ABI:
  * the chain sweep on flat tensors of 2^28 + 7 elements, lengths 1..32
    (random chains over add/mul/sigmoid/exp/relu/scale/cast, inputs U[-2,2]);
  * the same sweep preceded by ChannelShuffle(4) on fp16 [32,256,56,56];
  * residual add + RMSNorm + bf16 cast on [16384, 4096];
  * QKV split + transpose + RoPE on bf16 [32768, 3*32*128];
  * add -> relu -> scale on two fp32 vectors of 2^20;
  * the 3-scale detection-head decode into fp32 [1, 25200, 85].
`value` is the step's algorithmic minimum bytes (each input read once, each
output written once) divided by the device time of the step.  Inputs are
larger than L2 (the step streams ~29 GB, which evicts the two small
workloads' buffers between their uses).

Alongside: per-workload fused time and GB/s, the unfused per-op sequence
(one kernel per op with a full HBM round trip: the library's own length-1
chains for elementwise chains, PyTorch eager ops for the structured
workloads), the roofline of the dominant kernel, an end-to-end number with
host buffers, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-chain HBM GB/s (% of GB300 peak) and µs/chain vs unfused per-op"
UNIT = "GB/s"
WORKLOAD = ("all fused chains at full size: chain sweep L=1..32 on 2^28+7 elements and after "
            "ChannelShuffle(4) on fp16 [32,256,56,56]; ChannelShuffle(4) alone on the same "
            "tensor; RMSNorm+residual bf16 [16384,4096]; "
            "QKV split+RoPE bf16 [32768,3x32x128]; add-relu-scale fp32 2^20; detect decode "
            "3 scales fp16 -> fp32 [1,25200,85]")
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129e6  # GB300's L2, about 129 MB
LN_ROWS = [16384]  # rows of the LayerNorm next row ([4096] under --small)


# ---------------------------------------------------------------- helpers

def launch_overhead(t_unfused: float, t_fused: float, k: int):
    """Per-call fixed cost L and work T from the unfused time K*L + T and the
    fused time L + T (the launch-cost model of the NaiveRT analysis):
    L = (t_unfused - t_fused) / (K - 1), T = t_fused - L."""
    if k <= 1:
        return 0.0, t_fused
    L = (t_unfused - t_fused) / (k - 1)
    return L, t_fused - L


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed alone: the measured
    cuBLAS burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS burst)"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.2)
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workload

# Special-function unit (MUFU) work of a chain: exp is one ex2, sigmoid one
# ex2 and one rcp (the generated code's exp and sigmoid, accurate or fast).
# Rates per SM and clock: a probe of independent chains of each instruction
# on every SM of a GB300 measured ex2.approx at 9.5-9.9 T/s and rcp.approx at
# 4.8-5.0 T/s, 30-32 and 15-16 per SM-clock at 2.07 GHz: twice Blackwell's
# documented 16 for ex2, the same for rcp; an even mix of the two ran at 20,
# so they share one unit.  The floors take these at the sampled clock, or the
# rates every bench run measures with the library's own chains (mufu_rates)
# where those are higher, so that each floor stays a lower bound.
# With the HBM bytes this gives two lower bounds on a chain's time; chains
# heavy in the accurate exp and sigmoid can be bound by instruction issue
# instead, which is not modelled here.
EX2_PER_SM_CLK, RCP_PER_SM_CLK = 32, 16


def mufu_ops_per_element(spec):
    """(ex2, rcp) operations per element of a chain."""
    ops = [o.split(":")[0] for o in spec.split(";")]
    n_sig = ops.count("sigmoid")
    return ops.count("exp") + n_sig, n_sig


def mufu_floor_us(ops, rates):
    """Time the unit needs for (ex2, rcp) operations at rates (per second)."""
    return (ops[0] / rates["ex2_per_s"] + ops[1] / rates["rcp_per_s"]) * 1e6


def nominal_mufu_rates(sms, mhz):
    return {"ex2_per_s": EX2_PER_SM_CLK * sms * mhz * 1e6,
            "rcp_per_s": RCP_PER_SM_CLK * sms * mhz * 1e6,
            "source": f"{EX2_PER_SM_CLK} ex2 and {RCP_PER_SM_CLK} rcp per SM-clock at {mhz:.0f} MHz"}


def mufu_rates(dev, sms, mhz):
    """The special-function unit's ex2 and rcp rates, measured with the
    library's own kernels: a chain of 256 exp:fast (a multiply and an ex2
    each) and one of 128 sigmoid:fast (a multiply, an ex2, an add and an rcp)
    over 2^22 fp32 elements that stay in L2, 10 launches of each replayed
    from a graph.  The unit, not memory or issue, sets both times; the rcp
    rate is what the second leaves after its ex2s."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    n = 1 << 22
    x = W.device_uniform(n, -2.0, 2.0, 7, W.F32, dev)
    y = torch.empty_like(x)
    t = {}
    for name, op, k in (("exp", "exp:fast", 256), ("sigmoid", "sigmoid:fast", 128)):
        c = F.fuse_compile(";".join([op] * k), (n,), W.F32)
        t[name] = graph_per_launch(lambda c=c: F.fuse_launch(c, [x], y), k=10) / 1e3  # seconds
    ex2 = n * 256 / t["exp"]
    left = t["sigmoid"] / (n * 128) - 1.0 / ex2
    if left <= 0:
        raise RuntimeError("sigmoid chain no slower than its ex2s alone")
    rcp = 1.0 / left
    return {"ex2_per_s": ex2, "rcp_per_s": rcp, "ex2_per_sm_clk": ex2 / (sms * mhz * 1e6),
            "rcp_per_sm_clk": rcp / (sms * mhz * 1e6), "at_sm_mhz": mhz,
            "source": "measured: 256 exp:fast and 128 sigmoid:fast over 2^22 fp32 in L2"}


class Item:
    """One fused workload: a single launch of the library."""

    def __init__(self, name, nbytes, fused, unfused=None, n_unfused=0, kernel=None):
        self.name, self.bytes, self.fused = name, nbytes, fused
        self.unfused, self.n_unfused = unfused, n_unfused
        self.kernel = kernel
        self.inputs, self.outputs = [], []   # device tensors (for the end-to-end copies)
        # the same launch on other tensors of the same shapes (ins, outs)
        self.launch_on = None
        self.mufu_ops = None     # (ex2, rcp) special-function unit operations


def _tdt(dt):
    import torch
    return {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[dt]


def _esz(dt):
    return 4 if dt == 0 else 2


def build_items(dev, with_unfused=True, only=None, flat_elems=None, spec=None, spec_dtype=0):
    """The step's workloads; `only` (a regex) keeps the matching ones and
    `flat_elems` changes the flat chains' size (both for profiling a single
    kernel on a smaller case); `spec` replaces them all by one given chain."""
    import re

    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W

    items = []

    def want(name):
        return only is None or re.search(only, name) is not None

    def chain_item(name, spec, dt, shape, seed, lo=-2.0, hi=2.0, dev_inputs=None):
        n = int(np.prod(shape))
        c = F.fuse_compile(spec, shape, dt)
        ins = dev_inputs or [W.device_uniform(n, lo, hi, seed * 131 + j, d, dev)
                             for j, d in enumerate(c.in_dtypes)]
        out = torch.empty(n, dtype=_tdt(c.out_dtype), device=dev)
        nbytes = sum(n * _esz(d) for d in c.in_dtypes) + n * _esz(c.out_dtype)
        it = Item(name, nbytes, lambda: F.fuse_launch(c, ins, out), kernel=("chain", spec, shape, dt))
        it.inputs, it.outputs = ins, [out]
        it.launch_on = lambda i_s, o_s: F.fuse_launch(c, i_s, o_s[0])
        e, r = mufu_ops_per_element(spec)
        it.mufu_ops = (n * e, n * r) if e or r else None
        if with_unfused:
            it.unfused, it.n_unfused = unfused_chain(spec, dt, shape, ins, out)
        return it

    n_flat = flat_elems or W.FLAT_SIZES[-1]
    if spec is not None:  # one given chain, flat, as the only workload
        items.append(chain_item(f"chain[{spec}]_n{n_flat}", spec, spec_dtype, (n_flat,), 7))
        return items
    # chain sweep, flat, 2^28 + 7
    for L in W.CHAIN_LENGTHS:
        spec, dt = W.random_chain(L, 5)
        if want(f"flat_chain_L{L}_n{n_flat}"):
            items.append(chain_item(f"flat_chain_L{L}_n{n_flat}", spec, dt, (n_flat,), 100 + L))
    # chain sweep after ChannelShuffle(4), fp16 [32,256,56,56]
    cfg = W.SHUFFLE_CHAIN
    for L in W.CHAIN_LENGTHS:
        body, dt = W.random_chain(L, 9, start_dtype=W.F16)
        if want(f"shuffle_chain_L{L}"):
            items.append(chain_item(f"shuffle_chain_L{L}", f"shuffle:{cfg['groups']};{body}", dt,
                                    cfg["shape"], 200 + L))
    if want("channel_shuffle_g4_32x256x56x56_f16"):
        items.append(_shuffle_item(dev, with_unfused))
    if want(f"rmsnorm_residual_{W.RMSNORM['rows']}x{W.RMSNORM['hidden']}_bf16"):
        items.append(_rms_item(dev, with_unfused))
    if want(f"rope_qkv_split_{W.ROPE['tokens']}x{W.ROPE['heads']}x{W.ROPE['head_dim']}_bf16"):
        items.append(_rope_item(dev, with_unfused))
    ac = W.ADD_RELU_SCALE
    if want("add_relu_scale_1M_f32"):
        items.append(chain_item("add_relu_scale_1M_f32", ac["spec"], W.F32, (ac["n"],), ac["seed"],
                                ac["lo"], ac["hi"]))
    if want("detect_decode_3scale"):
        items.append(_detect_item(dev, with_unfused))
    return items


def _shuffle_item(dev, with_unfused):
    """ChannelShuffle alone through its entry point: a bit-exact permutation
    of whole H*W planes; unfused: PyTorch's view -> transpose -> contiguous."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    cfg = W.SHUFFLE_CHAIN
    n, c, h, w = cfg["shape"]
    g = cfg["groups"]
    x = W.device_uniform(n * c * h * w, cfg["lo"], cfg["hi"], 300, W.F16, dev)
    out = torch.empty_like(x)
    it = Item(f"channel_shuffle_g{g}_{n}x{c}x{h}x{w}_f16", 2 * x.numel() * 2,
              lambda: F.channel_shuffle(x, out, g, W.F16, shape=(n, c, h, w)),
              kernel=("chain", f"shuffle:{g}", cfg["shape"], W.F16))
    it.inputs, it.outputs = [x], [out]
    it.launch_on = lambda i_s, o_s: F.channel_shuffle(i_s[0], o_s[0], g, W.F16, shape=(n, c, h, w))
    if with_unfused:
        def unfused():
            return x.view(n, g, c // g, h, w).transpose(1, 2).contiguous().view(n, c, h, w)
        it.unfused, it.n_unfused = unfused, 1  # kernels, as --launch-trace counts them
    return it


def _rms_item(dev, with_unfused):
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    rc = W.RMSNORM
    rows, hidden = rc["rows"], rc["hidden"]
    x = W.device_normal((rows, hidden), 0, 1, rc["seed"], W.BF16, dev)
    r = W.device_normal((rows, hidden), 0, 1, rc["seed"] + 1, W.BF16, dev)
    w = W.device_normal((hidden,), 1, 0.1, rc["seed"] + 2, W.BF16, dev)
    y = torch.empty_like(x)
    ro = torch.empty_like(x)
    it = Item(f"rmsnorm_residual_{rows}x{hidden}_bf16", 4 * rows * hidden * 2 + hidden * 2,
              lambda: F.rmsnorm_residual(x, r, w, y, ro, rc["eps"], W.BF16),
              kernel=("rmsnorm",))
    it.inputs, it.outputs = [x, r, w], [y, ro]
    it.launch_on = lambda i_s, o_s: F.rmsnorm_residual(*i_s, *o_s, rc["eps"], W.BF16)
    if with_unfused:
        def rms_unfused():
            h = x + r
            hf = h.float()
            ms = hf.pow(2).mean(-1, keepdim=True)
            rstd = torch.rsqrt(ms + rc["eps"])
            return (hf * rstd * w.float()).to(torch.bfloat16), h
        it.unfused, it.n_unfused = rms_unfused, 10
    return it


def decode_glue(dev, layers=32, tokens=8, hidden=4096, heads=32, head_dim=128, ffn=11008,
                pos0=1000, reps=20):
    """The elementwise glue of a decoder's decode step, the multi-launch
    sequence "DeepJIT" section 6.1 measures per op, as a CUDA graph, and fused:
    per layer, residual + RMSNorm, QKV split + RoPE, a SwiGLU gate
    (sigmoid(g) * g * u as the chain sigmoid;mul;mul) and residual + RMSNorm
    again, at `tokens` tokens; the matrix products between them are not part of
    it.  Returns the time of one whole step (all layers), in microseconds,
    (a) as PyTorch eager ops, (b) those replayed from one CUDA graph, (c) the
    library's fused calls from a host loop, (d) those replayed from one
    library graph."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    bf = torch.bfloat16
    x = [W.device_normal((tokens, hidden), 0, 1, 900 + i, W.BF16, dev) for i in range(layers)]
    r = [W.device_normal((tokens, hidden), 0, 1, 1000 + i, W.BF16, dev) for i in range(layers)]
    wn = W.device_normal((hidden,), 1, 0.1, 1100, W.BF16, dev)
    qkv = [W.device_normal((tokens, 3 * heads * head_dim), 0, 1, 1200 + i, W.BF16, dev)
           for i in range(layers)]
    gate = [W.device_normal((tokens, ffn), 0, 1, 1300 + i, W.BF16, dev) for i in range(layers)]
    up = [W.device_normal((tokens, ffn), 0, 1, 1400 + i, W.BF16, dev) for i in range(layers)]
    y, ro = torch.empty_like(x[0]), torch.empty_like(x[0])
    y2, ro2 = torch.empty_like(x[0]), torch.empty_like(x[0])
    q, k, v = (torch.empty(heads * tokens * head_dim, dtype=bf, device=dev) for _ in range(3))
    act = torch.empty_like(gate[0])
    swiglu = F.fuse_compile("sigmoid;mul;mul", (tokens, ffn), W.BF16)
    stream = torch.cuda.Stream()

    def fused():
        for i in range(layers):
            F.rmsnorm_residual(x[i], r[i], wn, y, ro, 1e-6, W.BF16, stream=stream)
            F.rope_qkv_split(qkv[i], q, k, v, heads, head_dim, pos0, 10000.0, W.BF16,
                             stream=stream)
            F.fuse_launch(swiglu, [gate[i], gate[i], up[i]], act, stream=stream)
            F.rmsnorm_residual(ro, x[i], wn, y2, ro2, 1e-6, W.BF16, stream=stream)

    pos = torch.arange(pos0, pos0 + tokens, device=dev, dtype=torch.float64)
    inv = 10000.0 ** (-torch.arange(0, head_dim, 2, device=dev, dtype=torch.float64) / head_dim)
    ang = pos[:, None] * inv[None, :]
    cos = torch.cat([ang.cos(), ang.cos()], -1).float()[None]
    sin = torch.cat([ang.sin(), ang.sin()], -1).float()[None]

    def rms(a, b):
        h = a.float() + b.float()
        return (h * torch.rsqrt(h.pow(2).mean(-1, keepdim=True) + 1e-6) * wn.float()).to(bf), \
            h.to(bf)

    def eager():
        for i in range(layers):
            yy, hh = rms(x[i], r[i])
            t = qkv[i].view(tokens, 3, heads, head_dim)
            outs = [t[:, j].transpose(0, 1).contiguous() for j in range(3)]
            for j in range(2):
                xf = outs[j].float()
                rh = torch.cat([-xf[..., head_dim // 2:], xf[..., :head_dim // 2]], -1)
                outs[j] = (xf * cos + rh * sin).to(bf)
            gf = gate[i].float()
            a_ = (torch.sigmoid(gf) * gf * up[i].float()).to(bf)
            rms(hh, x[i])

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            for _ in range(reps):
                fn()
            b.record()
        b.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    out = {"layers": layers, "tokens": tokens, "launches_fused": 4 * layers,
           "us_eager": timed(eager), "us_fused_host_loop": timed(fused)}
    # the same sequences replayed from one graph each
    with torch.cuda.stream(stream):
        eager()
    stream.synchronize()
    tg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tg, stream=stream):
        eager()
    out["us_eager_graph"] = timed(tg.replay)
    F.fuse_graph_begin(stream)
    with torch.cuda.stream(stream):
        fused()
    g = F.fuse_graph_end(stream)
    out["us_fused_graph"] = timed(lambda: g.launch(stream))
    out["graph_nodes_fused"] = g.nodes
    g.release()
    return out


def _ln_item(dev, with_unfused):
    """Residual add + LayerNorm (a next row, measured beside the step)."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    rows, hidden, eps = LN_ROWS[0], 4096, 1e-5
    x = W.device_normal((rows, hidden), 0, 1, 61, W.BF16, dev)
    r = W.device_normal((rows, hidden), 0, 1, 62, W.BF16, dev)
    g = W.device_normal((hidden,), 1, 0.1, 63, W.BF16, dev)
    b = W.device_normal((hidden,), 0, 0.1, 64, W.BF16, dev)
    y, ro = torch.empty_like(x), torch.empty_like(x)
    it = Item(f"layernorm_residual_{rows}x{hidden}_bf16", 4 * rows * hidden * 2 + 2 * hidden * 2,
              lambda: F.layernorm_residual(x, r, g, b, y, ro, eps, W.BF16), kernel=("layernorm",))
    it.inputs, it.outputs = [x, r, g, b], [y, ro]
    it.launch_on = lambda i_s, o_s: F.layernorm_residual(*i_s, *o_s, eps, W.BF16)
    if with_unfused:
        def ln_unfused():
            h = x + r
            hf = h.float()
            mean = hf.mean(-1, keepdim=True)
            d = hf - mean
            var = (d * d).mean(-1, keepdim=True)
            return (d * torch.rsqrt(var + eps) * g.float() + b.float()).to(torch.bfloat16), h
        it.unfused, it.n_unfused = ln_unfused, 14  # kernels, as --launch-trace counts them
    return it


def _rms_linear_item(dev, with_unfused, M=16384):
    """RMSNorm -> Linear -> scale on the tensor cores (a next row, measured
    beside the step); unfused: the PyTorch RMSNorm ops, then F.linear
    (cuBLAS), then the scale."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    N, K, eps, scale = 4096, 4096, 1e-6, 0.5
    x = W.device_normal((M, K), 0, 1, 71, W.BF16, dev)
    g = W.device_normal((K,), 1, 0.1, 72, W.BF16, dev)
    w = W.device_normal((N, K), 0, K ** -0.5, 73, W.BF16, dev)
    b = W.device_normal((N,), 0, 0.5, 74, W.BF16, dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wf = torch.empty_like(w)  # gamma folded into the weight once, like loading weights
    F.rmsnorm_linear_fold(w, g, wf, W.BF16)
    it = Item(f"rmsnorm_linear_{M}x{N}x{K}_bf16", 2 * (M * K + N * K + M * N),
              lambda: F.rmsnorm_linear(x, None, wf, b, out, eps, scale, W.BF16),
              kernel=("rms_linear",))
    it.flops = 2 * M * N * K
    it.inputs, it.outputs = [x, g, w, b], [out]
    if with_unfused:
        def unfused():
            xf = x.float()
            y = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps) * g.float()).to(torch.bfloat16)
            return torch.nn.functional.linear(y, w, b) * scale
        it.unfused, it.n_unfused = unfused, 11  # kernels, as --launch-trace counts them
        # the bare GEMM of the same shape in the vendor library, no norm, no
        # bias, no scale: what the fused kernel's contraction is held against
        gemm_out = torch.empty_like(out)
        it.library_gemm = lambda: torch.matmul(x, wf.t(), out=gemm_out)
    # gamma passed per call: folded into stream-ordered scratch, then the product
    it.gamma_path = lambda: F.rmsnorm_linear(x, g, w, b, out, eps, scale, W.BF16)
    return it


def fast_math_row(dev, peak, peak_kind, rates):
    """The shuffle-prefixed 16-op chain (4 exp, 4 sigmoid) with its exp and
    sigmoid in the opt-in fast form (exp:fast, sigmoid:fast: ex2.approx on
    x * log2 e, validated against the oracle's bound for it) beside the
    accurate form, each timed as the step's workloads are on their own
    (steady_times)."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    cfg = W.SHUFFLE_CHAIN
    body, dt = W.random_chain(16, 9, start_dtype=W.F16)
    fast = ";".join("exp:fast" if o == "exp" else "sigmoid:fast" if o == "sigmoid" else o
                    for o in body.split(";"))
    n = int(np.prod(cfg["shape"]))
    out = {}
    for tag, spec in (("accurate", body), ("fast", fast)):
        c = F.fuse_compile(f"shuffle:{cfg['groups']};{spec}", cfg["shape"], dt)
        ins = [W.device_uniform(n, -2.0, 2.0, 200 + 16 + j, d, dev) for j, d in enumerate(c.in_dtypes)]
        o = torch.empty(n, dtype=_tdt(c.out_dtype), device=dev)
        nb = sum(n * _esz(d) for d in c.in_dtypes) + n * _esz(c.out_dtype)
        it = Item(tag, nb, None)
        it.inputs, it.outputs = ins, [o]
        it.launch_on = lambda i_s, o_s, c=c: F.fuse_launch(c, i_s, o_s[0])
        out["us_" + tag] = steady_times(it, 60)[0]
        del it, ins, o
    e, r = mufu_ops_per_element(body)
    mufu_us = mufu_floor_us((n * e, n * r), rates)
    hbm_us = nb / (peak * 1e9) * 1e6
    out.update({"bytes": nb, "spec_fast": fast, "mufu_bound_us": mufu_us, "hbm_bound_us": hbm_us,
                "bound": "mufu" if mufu_us > hbm_us else "hbm",
                "frac_of_bound_fast": max(mufu_us, hbm_us) / out["us_fast"],
                "frac_of_bound_accurate": max(mufu_us, hbm_us) / out["us_accurate"]})
    return {"shuffle_chain_L16_fast_math": out}


def noalloc_row(dev, peak, peak_kind):
    """rope_qkv_split_noalloc at the most tokens its fixed array takes at
    head_dim 128 (8192 x 32 heads, bf16), beside rope_qkv_split on the same
    tensors: its two launches (the cos/sin rows, then the rotation) against
    the generated kernel with the library's cached table."""
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    T, H, D = 8192, 32, 128
    qkv = W.device_normal((T, 3 * H * D), 0, 1, 81, W.BF16, dev)
    q, k, v = (torch.empty(H * T * D, dtype=torch.bfloat16, device=dev) for _ in range(3))
    nb = 2 * T * 3 * H * D * 2
    ms = time_fn(lambda: F.rope_qkv_split_noalloc(qkv, q, k, v, H, D, 0, 10000.0, W.BF16),
                 reps=20, warm=3)
    ref = time_fn(lambda: F.rope_qkv_split(qkv, q, k, v, H, D, 0, 10000.0, W.BF16), reps=20, warm=3)
    return {f"rope_qkv_split_noalloc_{T}x{H}x{D}_bf16": {
        "bytes": nb, "us_fused": ms * 1e3, "gbs": nb / (ms / 1e3) / 1e9,
        "frac_of_" + peak_kind + "_peak": nb / (ms / 1e3) / 1e9 / peak, "launches": 2,
        "us_rope_qkv_split_same_shape": ref * 1e3}}


def _rope_item(dev, with_unfused):
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    pc = W.ROPE
    T, H, D = pc["tokens"], pc["heads"], pc["head_dim"]
    qkv = W.device_normal((T, 3 * H * D), 0, 1, pc["seed"], W.BF16, dev)
    q, k, v = (torch.empty(H * T * D, dtype=torch.bfloat16, device=dev) for _ in range(3))
    it = Item(f"rope_qkv_split_{T}x{H}x{D}_bf16", 2 * T * 3 * H * D * 2,
              lambda: F.rope_qkv_split(qkv, q, k, v, H, D, pc["pos0"], pc["base"], W.BF16),
              kernel=("rope",))
    it.inputs, it.outputs = [qkv], [q, k, v]
    it.launch_on = lambda i_s, o_s: F.rope_qkv_split(i_s[0], *o_s, H, D, pc["pos0"], pc["base"],
                                                     W.BF16)
    if with_unfused:
        pos = torch.arange(T, device=dev, dtype=torch.float64)
        inv = pc["base"] ** (-torch.arange(0, D, 2, device=dev, dtype=torch.float64) / D)
        ang = pos[:, None] * inv[None, :]
        cos = torch.cat([ang.cos(), ang.cos()], -1).float()
        sin = torch.cat([ang.sin(), ang.sin()], -1).float()

        def rope_unfused():
            t = qkv.view(T, 3, H, D)
            outs = [t[:, i].transpose(0, 1).contiguous() for i in range(3)]
            for i in range(2):
                xf = outs[i].float()
                rh = torch.cat([-xf[..., D // 2:], xf[..., :D // 2]], -1)
                outs[i] = (xf * cos + rh * sin).to(torch.bfloat16)
            return outs
        it.unfused, it.n_unfused = rope_unfused, 17  # kernels, as --launch-trace counts them
    return it


def _detect_item(dev, with_unfused):
    import torch

    import elementwise_chain_jit_gb300 as F
    import workloads as W
    dc = W.DETECT
    anchors = W.detect_anchors(dc["strides"], dc["na"])
    feats = [W.device_normal((1, dc["na"] * dc["no"], h, w_), 0, dc["sd"], dc["seed"] + s, W.F16, dev)
             for s, (h, w_) in enumerate(dc["hw"])]
    nrows = sum(dc["na"] * h * w_ for h, w_ in dc["hw"])
    dout = torch.empty(nrows * dc["no"], dtype=torch.float32, device=dev)
    # the fixed arguments converted once, as a caller decoding every frame would
    dec = F.DetectDecoder(dc["hw"], dc["strides"], anchors, dc["na"], dc["no"], W.F16)
    it = Item("detect_decode_3scale", sum(f.numel() * 2 for f in feats) + dout.numel() * 4,
              lambda: dec(feats, dout),
              kernel=("detect",))
    it.inputs, it.outputs = feats, [dout]
    it.launch_on = lambda i_s, o_s: dec(i_s, o_s[0])
    if with_unfused:
        an = torch.tensor(anchors, dtype=torch.float32, device=dev)
        grids = []
        for h, w_ in dc["hw"]:
            yy, xx = torch.meshgrid(torch.arange(h, device=dev), torch.arange(w_, device=dev),
                                    indexing="ij")
            grids.append(torch.stack([xx, yy], -1).float().view(1, 1, h, w_, 2))

        def detect_unfused():
            outs = []
            for s, (h, w_) in enumerate(dc["hw"]):
                xs = feats[s].view(1, dc["na"], dc["no"], h, w_).permute(0, 1, 3, 4, 2).contiguous()
                p = xs.float().sigmoid()
                xy = (p[..., :2] * 2 - 0.5 + grids[s]) * dc["strides"][s]
                wh = (p[..., 2:4] * 2) ** 2 * an[s].view(1, dc["na"], 1, 1, 2)
                outs.append(torch.cat([xy, wh, p[..., 4:]], -1).view(1, -1, dc["no"]))
            return torch.cat(outs, 1)
        it.unfused, it.n_unfused = detect_unfused, 40  # kernels, as --launch-trace counts them
    return it


def unfused_chain(spec, dt, shape, ins, out):
    """The same chain as one library kernel per op, each writing a full
    intermediate tensor in the chain's current dtype."""
    import torch

    import elementwise_chain_jit_gb300 as F
    steps = []
    n = int(np.prod(shape))
    cur_dt, j = dt, 1
    bufs = {}

    def buf(d, slot):
        key = (d, slot)
        if key not in bufs:
            bufs[key] = torch.empty(n, dtype=_tdt(d), device=out.device)
        return bufs[key]

    items = [s.strip() for s in spec.split(";") if s.strip()]
    src = ins[0]
    slot = 0
    for pos, item in enumerate(items):
        name, _, arg = item.partition(":")
        if name == "shuffle":
            c = F.fuse_compile(item, shape, cur_dt)
            operands = [src]
        elif name in ("add", "mul"):
            c = F.fuse_compile(name, (n,), cur_dt)
            operands = [src, ins[j]]
            j += 1
        else:
            c = F.fuse_compile(item, (n,), cur_dt)
            operands = [src]
        if name == "cast":
            cur_dt = {"f32": 0, "f16": 1, "bf16": 2}[arg]
        last = pos == len(items) - 1
        dst = out if last else buf(cur_dt, slot)
        slot ^= 1
        steps.append((c, list(operands), dst))
        src = dst
    if not items:
        return None, 0

    def run():
        for c, operands, dst in steps:
            F.fuse_launch(c, operands, dst)
    return run, len(steps)


# ---------------------------------------------------------------- timing

def time_fn(fn, reps=5, warm=2):
    import torch
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def graph_per_launch(fn, k=20):
    """Device time per launch of fn, from k launches captured into one library
    graph and replayed once (no host cost between launches)."""
    import torch

    import elementwise_chain_jit_gb300 as F
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
    s.synchronize()
    F.fuse_graph_begin(s)
    with torch.cuda.stream(s):
        for _ in range(k):
            fn()
    g = F.fuse_graph_end(s)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.launch(s)
        s.synchronize()
        a.record(s)
        g.launch(s)
        b.record(s)
        b.synchronize()
    g.release()
    return a.elapsed_time(b) / k


def steady_times(item, launches):
    """One workload launched back to back on its own, `launches` times, on
    rotating buffer sets: its own tensors and copies of them, enough sets that
    together they exceed twice the L2, so every launch reads its inputs from
    HBM and the dirty lines one launch leaves drain during the next ones, as
    in any pipeline.  The launches are captured into one library graph (from
    the host a few-microsecond kernel would wait on its own launch) and
    replayed with launch-order overlap intact and no event between them.
    Returns (mean us a launch from events around one replay, per-launch us
    from the CUPTI trace of another -- end of a kernel minus the end of the
    one before, the first launch left out -- or None where the trace does not
    hold one kernel per launch)."""
    import torch
    from torch.profiler import ProfilerActivity, profile

    import elementwise_chain_jit_gb300 as F
    nsets = 1 if item.bytes >= 2 * L2_BYTES else int(2 * L2_BYTES // item.bytes) + 2
    sets = [(item.inputs, item.outputs)]
    sets += [([t.clone() for t in item.inputs], [torch.empty_like(t) for t in item.outputs])
             for _ in range(nsets - 1)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i_s, o_s in sets:
            item.launch_on(i_s, o_s)
    s.synchronize()
    F.fuse_graph_begin(s)
    with torch.cuda.stream(s):
        for k in range(launches):
            item.launch_on(*sets[k % nsets])
    g = F.fuse_graph_end(s)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.launch(s)
    s.synchronize()
    a.record(s)
    g.launch(s)
    b.record(s)
    b.synchronize()
    mean_us = a.elapsed_time(b) / launches * 1e3
    # a third replay under the trace (which adds its own cost to the replay)
    device_ops(lambda: None)  # the process's first session can miss records
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        g.launch(s)
        s.synchronize()
    g.release()
    ends = sorted((e.start_ns() + e.duration_ns()) / 1e3 for e in prof.profiler.kineto_results.events()
                  if e.device_type() == torch.autograd.DeviceType.CUDA)
    per = None
    if len(ends) == launches:
        per = [ends[i] - ends[i - 1] for i in range(1, launches)]
    del sets
    return mean_us, per


def cold_time(item, reps=10):
    """Mean time of one launch with its inputs cold in HBM and no dirty lines
    left in L2: before each launch a read-only pass over 512 MB (four times
    L2) evicts L2 with clean lines.  The mean, not the median: on these boxes
    an event pair around one launch reads in steps of about 2.05 us, and the
    launch starts at a random point of that step (after a flush pass of
    varying length), so the mean of many launches is unbiased where the
    median is not."""
    import torch
    flush = getattr(cold_time, "buf", None)
    if flush is None:
        flush = cold_time.buf = torch.ones(128 << 20, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    ts = []
    for _ in range(reps + 2):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        item.fused()
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts[2:]) * 1e3


def graph_times(item, k=50):
    """Launch overhead of a small workload ("DeepJIT" section 6.1's per-op /
    CUDA graph / fused comparison): mean time per pass over k passes of
    (a) the fused launch from the host, (b) the fused launch replayed from one
    library graph, (c) the unfused sequence replayed from one CUDA graph.
    Inputs stay in L2 across the k passes (warm)."""
    import torch

    import elementwise_chain_jit_gb300 as F
    s = torch.cuda.Stream()
    out = {}
    with torch.cuda.stream(s):
        item.fused()
        s.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(k):
            item.fused()
        b.record(s)
        b.synchronize()
        out["us_fused_host_loop"] = a.elapsed_time(b) / k * 1e3
    F.fuse_graph_begin(s)
    with torch.cuda.stream(s):
        for _ in range(k):
            item.fused()
    g = F.fuse_graph_end(s)
    with torch.cuda.stream(s):
        g.launch(s)
        s.synchronize()
        a.record(s)
        g.launch(s)
        b.record(s)
        b.synchronize()
    out["us_fused_graph"] = a.elapsed_time(b) / k * 1e3
    g.release()
    if item.unfused is not None:
        with torch.cuda.stream(s):
            item.unfused()
        s.synchronize()
        tg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tg, stream=s):
            for _ in range(k):
                item.unfused()
        tg.replay()
        torch.cuda.synchronize()
        a.record()
        tg.replay()
        b.record()
        b.synchronize()
        out["us_unfused_graph"] = a.elapsed_time(b) / k * 1e3
    return out


_LATENCY_CHILD = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import elementwise_chain_jit_gb300 as F
F.fuse_device_sms()  # driver and context up before anything is timed
t0 = time.perf_counter()
c = F.fuse_compile({spec!r}, ({n},), {dt})
t1 = time.perf_counter()
c2 = F.fuse_compile({spec!r}, ({n},), {dt})
t2 = time.perf_counter()
print(json.dumps(dict(F.fuse_stats(), first_ms=(t1 - t0) * 1e3, again_ms=(t2 - t1) * 1e3)))
"""


def compile_latency(spec, n, dt):
    """First-call latency of fuse_compile for one chain ("DeepJIT", section
    6.2: the compile cache keeps NVRTC off the request path): a fresh process
    with an empty cache directory (NVRTC compile + module load), a second
    fresh process on the same directory (disk hit + module load), and a
    second call in that process (memory hit).  Each first call is preceded by
    the driver and context set-up, which is not timed."""
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        env = dict(os.environ, FUSE_CACHE_DIR=d)
        env.pop("FUSE_NVRTC_OPTIONS", None)
        code = _LATENCY_CHILD.format(root=ROOT, spec=spec, n=n, dt=dt)
        runs = []
        for _ in range(2):
            r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                               text=True, timeout=600)
            if r.returncode != 0:
                return {"error": r.stderr.strip().splitlines()[-1:]}
            runs.append(json.loads(r.stdout.strip().splitlines()[-1]))
    cold, disk = runs
    return {"spec": spec, "n": n, "cold_nvrtc_ms": cold["first_ms"], "cold_compiles": cold["compiles"],
            "disk_hit_ms": disk["first_ms"], "disk_compiles": disk["compiles"],
            "memory_hit_ms": disk["again_ms"],
            "note": "first fuse_compile in a fresh process, driver and context already up; "
                    "cold and disk include loading the module on the GPU"}


def kernel_source_hash(item):
    import elementwise_chain_jit_gb300 as F
    h = hashlib.sha1()
    if item.kernel and item.kernel[0] == "chain":
        _, spec, shape, dt = item.kernel
        h.update(F.fuse_source(spec, shape, dt).encode())
        h.update(open(os.path.join(ROOT, "elementwise_chain_jit_gb300", "csrc", "kernels",
                                   "common.cuh"), "rb").read())
    else:
        for f in ("common.cuh", f"{item.kernel[0]}.cuh"):
            p = os.path.join(ROOT, "elementwise_chain_jit_gb300", "csrc", "kernels", f)
            if os.path.exists(p):
                h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_record(name, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (lines 'kernel: <name> source: <hash> traffic_bytes: <B>')."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 6 and parts[0] == "kernel:" and parts[1] == name and parts[3] == src_hash:
            return float(parts[5])
    return None


# ---------------------------------------------------------------- CPU oracle baseline

def cpu_sample_all_cores(frac_div: int):
    """The flat-chain part of the sample on every host core: the elements split
    into one contiguous slice per core, one thread each, the same oracle call
    per slice (ctypes releases the GIL while the C oracle runs).  Returns
    (bytes, seconds, threads, description)."""
    import concurrent.futures as cf

    import oracle
    import workloads as W
    cores = os.cpu_count() or 1
    n = W.FLAT_SIZES[-1] // frac_div
    bounds = np.linspace(0, n, cores + 1).astype(np.int64)
    total_b, total_t = 0, 0.0
    with cf.ThreadPoolExecutor(cores) as ex:
        for L in W.CHAIN_LENGTHS:
            spec, dt = W.random_chain(L, 5)
            ins, dts = W.chain_inputs(spec, dt, n, L)
            ch = oracle.parse_spec(spec, dt)

            def part(i, spec=spec, dt=dt, ins=ins, ch=ch):
                lo, hi = int(bounds[i]), int(bounds[i + 1])
                vals = oracle.chain_eval(spec, dt, [a[lo:hi] for a in ins], (hi - lo,))[0]
                return oracle.store(vals, ch.out_dtype)
            t0 = time.perf_counter()
            list(ex.map(part, range(cores)))
            total_t += time.perf_counter() - t0
            total_b += sum(n * _esz(d) for d in dts) + n * _esz(ch.out_dtype)
    return total_b, total_t, cores, f"flat chains L=1..32 on {n} elements, {cores} slices, one thread each"


def sample_share(frac_div: int) -> str:
    """What share of each workload cpu_sample(frac_div) runs: the shuffle
    workloads shrink by whole batches only, detect by whole cells per side."""
    nb = 32 // min(frac_div, 32)
    return (f"1/{frac_div} of the flat chains, RMSNorm, RoPE and add-relu-scale; "
            f"{nb}/32 of the shuffle workloads' batch; detect with each scale's sides "
            f"divided by {int(np.sqrt(frac_div))}, at least 1 cell")


def cpu_sample(frac_div: int):
    """The oracle on a bounded sample of every workload; returns (bytes, seconds, description)."""
    import oracle
    import workloads as W
    total_b, total_t, parts = 0, 0.0, []

    def clock(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    n = W.FLAT_SIZES[-1] // frac_div
    for L in W.CHAIN_LENGTHS:
        spec, dt = W.random_chain(L, 5)
        ins, dts = W.chain_inputs(spec, dt, n, L)
        ch = oracle.parse_spec(spec, dt)
        total_t += clock(lambda: oracle.store(oracle.chain_eval(spec, dt, ins, (n,))[0], ch.out_dtype))
        total_b += sum(n * _esz(d) for d in dts) + n * _esz(ch.out_dtype)
    parts.append(f"flat chains L=1..32 on {n} elements")
    cfg = W.SHUFFLE_CHAIN
    nb = max(1, cfg["shape"][0] // min(frac_div, cfg["shape"][0]))
    shape = (nb,) + tuple(cfg["shape"][1:])
    ns = int(np.prod(shape))
    for L in W.CHAIN_LENGTHS:
        body, dt = W.random_chain(L, 9, start_dtype=W.F16)
        spec = f"shuffle:{cfg['groups']};{body}"
        ins, dts = W.chain_inputs(spec, dt, ns, L)
        ch = oracle.parse_spec(spec, dt)
        total_t += clock(lambda: oracle.store(oracle.chain_eval(spec, dt, ins, shape)[0], ch.out_dtype))
        total_b += sum(ns * _esz(d) for d in dts) + ns * _esz(ch.out_dtype)
    parts.append(f"shuffle chains L=1..32 on batch {nb} of [32,256,56,56]")
    xs = W.uniform(ns, cfg["lo"], cfg["hi"], 300, W.F16).reshape(shape)
    total_t += clock(lambda: oracle.channel_shuffle(xs, cfg["groups"]))
    total_b += 2 * ns * 2
    parts.append(f"channel shuffle on batch {nb}")
    rc = W.RMSNORM
    rows = max(1, rc["rows"] // frac_div)
    x = W.normal((rows, rc["hidden"]), 0, 1, 1, W.BF16)
    r = W.normal((rows, rc["hidden"]), 0, 1, 2, W.BF16)
    w = W.normal(rc["hidden"], 1, 0.1, 3, W.BF16)

    def rms():
        y, h = oracle.rmsnorm_residual(x, r, w, W.BF16, rc["eps"])
        oracle.store(y, W.BF16), oracle.store(h, W.BF16)
    total_t += clock(rms)
    total_b += 4 * rows * rc["hidden"] * 2 + rc["hidden"] * 2
    parts.append(f"rmsnorm {rows} rows")
    pc = W.ROPE
    toks = max(1, pc["tokens"] // frac_div)
    qkv = W.normal((toks, 3 * pc["heads"] * pc["head_dim"]), 0, 1, 4, W.BF16)

    def rope():
        q, k, v, _, _ = oracle.rope_qkv_split(qkv, W.BF16, pc["heads"], pc["head_dim"], np.arange(toks))
        for a in (q, k, v):
            oracle.store(a, W.BF16)
    total_t += clock(rope)
    total_b += 2 * qkv.size * 2
    parts.append(f"rope {toks} tokens")
    ac = W.ADD_RELU_SCALE
    na = max(1, ac["n"] // frac_div)
    a = W.uniform(na, -1, 1, 5, W.F32)
    b = W.uniform(na, -1, 1, 6, W.F32)
    total_t += clock(lambda: oracle.store(oracle.chain_eval(ac["spec"], W.F32, [a, b], (na,))[0], W.F32))
    total_b += 3 * na * 4
    parts.append(f"add-relu-scale {na} elements")
    dc = W.DETECT
    hw = [(max(1, h // int(np.sqrt(frac_div))), max(1, w_ // int(np.sqrt(frac_div)))) for h, w_ in dc["hw"]]
    feats = [W.normal((1, 255, h, w_), 0, 2, 7 + s, W.F16) for s, (h, w_) in enumerate(hw)]
    anchors = W.detect_anchors(dc["strides"])
    total_t += clock(lambda: oracle.detect_decode(feats, W.F16, dc["strides"], anchors, 3, 85))
    total_b += sum(f.size * 2 for f in feats) + sum(3 * h * w_ for h, w_ in hw) * 85 * 4
    parts.append(f"detect decode scales {hw}")
    return total_b, total_t, "; ".join(parts)


# ---------------------------------------------------------------- arms

def max_over_ranks(local_ms: float, world: int, device=None) -> float:
    """The job's time: the slowest rank's (every rank runs its own full step)."""
    if world <= 1:
        return local_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's step bytes over the slowest step."""
    return world * step_bytes / (ms_per_step / 1e3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    frac = 1024
    for _ in range(args.warmup):
        cpu_sample(frac)
    tb, tt = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        b, t, desc = cpu_sample(frac)
        tb += b
        tt += t
    v = tb / tt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample_share(frac) + " per step"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import re

    import torch

    import elementwise_chain_jit_gb300 as F

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    items = build_items(dev, with_unfused=not args.no_unfused, only=args.only,
                        flat_elems=args.flat_elems, spec=args.spec,
                        spec_dtype={"f32": 0, "f16": 1, "bf16": 2}[args.spec_dtype])
    if not items:
        raise SystemExit(f"--only {args.only!r} matches no workload")
    if args.launch_trace:
        return run_launch_trace(args, items, dev)
    if args.sequences_once:
        return run_sequences_once(args, items, dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    step_bytes = sum(it.bytes for it in items)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up (compiles and loads everything)
    for _ in range(args.warmup):
        for it in items:
            it.fused()
    barrier()
    # Timed region: K steps of back-to-back launches.  An event recorded
    # between two launches makes the second wait for the first to finish
    # before it is launched, which undoes programmatic dependent launch (about
    # 4.6 us a launch, measured); so inside the timed region events bracket
    # only the dominant kernel -- the workload with the most algorithmic
    # bytes, whose duration the roofline needs.  Every workload's own time
    # comes from a second pass of K steps with an event between every two
    # launches (per_chain; each of those times includes a launch gap).
    nitem = len(items)
    dom = max(range(nitem), key=lambda i: items[i].bytes)
    ev_dom = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    launches0 = F.fuse_stats()["launches"]
    with ClockSampler(local) as clocks:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            for i, it in enumerate(items):
                if i == dom:
                    ev_dom[s][0].record(stream)
                it.fused()
                if i == dom:
                    ev_dom[s][1].record(stream)
        t_end.record(stream)
        barrier()
    launches = F.fuse_stats()["launches"] - launches0
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    dom_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_dom)
    ms_per_step = total_ms / args.steps
    value = job_gbs(step_bytes, world, ms_per_step)
    # attribution pass (outside the timed region): an event between every two
    # launches gives each workload's time in the step
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nitem + 1)] for _ in range(args.steps)]
    barrier()
    for s in range(args.steps):
        evs[s][0].record(stream)
        for i, it in enumerate(items):
            it.fused()
            evs[s][i + 1].record(stream)
    barrier()
    per_step = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps)]
                for i in range(nitem)]
    per_item = [statistics.mean(t) for t in per_step]
    ms_per_step_item_events = sum(per_item)
    # and each workload's cost in the undisturbed pipeline, from kernel end times
    pipe, pipe_step_us = None, None
    if world == 1:
        try:
            pipe, pipe_step_us = pipeline_times(items, min(args.steps, 20))
        except Exception as e:  # a profiler that cannot start leaves the figure out
            print(f"pipeline attribution skipped: {e}", file=sys.stderr)

    peak, peak_kind = peaks()
    # the special-function unit's rates, for the chains' second floor
    mhz = clocks.summary().get("sm_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rates = nominal_mufu_rates(sms, mhz)
    mufu_report = {"floor": rates}
    if any(it.mufu_ops for it in items) or args.only is None or re.search(args.only, "fast_math"):
        try:
            measured = mufu_rates(dev, sms, mhz)
            mufu_report["measured"] = measured
            if measured["ex2_per_s"] > rates["ex2_per_s"] or measured["rcp_per_s"] > rates["rcp_per_s"]:
                rates = {"ex2_per_s": max(rates["ex2_per_s"], measured["ex2_per_s"]),
                         "rcp_per_s": max(rates["rcp_per_s"], measured["rcp_per_s"]),
                         "source": "the larger of the per-clock rates and the measured ones"}
                mufu_report["floor"] = rates
        except Exception as e:  # the floors keep the per-clock rates
            mufu_report["measured"] = {"error": str(e)[:200]}
    # unfused per-op sequences (outside the timed region)
    per_chain = {}
    for it, ems, ts in zip(items, per_item, per_step):
        # the workload's own figure: back to back on rotating buffer sets
        st_us, st_per = steady_times(it, 60 if it.bytes < 1e9 else 10)
        ms = st_us / 1e3
        d = {"bytes": it.bytes, "us_fused": st_us, "gbs": it.bytes / (ms / 1e3) / 1e9,
             "frac_of_" + peak_kind + "_peak": it.bytes / (ms / 1e3) / 1e9 / peak}
        if st_per:
            q = np.percentile(st_per, [10, 50, 90])
            d.update({"us_p10": q[0], "us_median": q[1], "us_p90": q[2]})
        # inside the step, an event between every two launches
        q = np.percentile(ts, [10, 50, 90])
        d.update({"us_in_step_events": ems * 1e3,
                  "frac_in_step_events": it.bytes / (ems / 1e3) / 1e9 / peak,
                  "us_in_step_events_p10_p50_p90": [q[0] * 1e3, q[1] * 1e3, q[2] * 1e3]})
        if pipe:
            d.update({"us_in_pipeline": pipe[it.name],
                      "frac_in_pipeline": it.bytes / (pipe[it.name] * 1e-6) / 1e9 / peak})
        if it.unfused is not None and not args.no_unfused:
            ums = time_fn(it.unfused, reps=3, warm=1)
            L, T = launch_overhead(ums, ms, it.n_unfused)
            d.update({"us_unfused": ums * 1e3, "unfused_kernels": it.n_unfused,
                      "speedup": ums / ms, "extra_cost_per_unfused_op_us": L * 1e3})
        if it.bytes < 64e6 and not args.no_unfused:
            d.update(graph_times(it))
        # the same launch alone, inputs cold and no predecessor's dirty lines
        # left in L2 to write back (in the step each item pays for those)
        cold_us = cold_time(it, reps=40 if it.bytes < 1e9 else 5)
        d.update({"us_fused_cold_clean_l2": cold_us,
                  "frac_cold_clean_l2": it.bytes / (cold_us * 1e-6) / 1e9 / peak})
        if it.name.startswith("channel_shuffle"):
            # the same bytes through PyTorch's device-to-device copy, timed the
            # same way: what a plain copy of this size reaches on this machine
            src, dst = it.inputs[0], it.outputs[0]

            class _Copy:
                fused = staticmethod(lambda: dst.copy_(src))
            copy_us = cold_time(_Copy, reps=40)
            d.update({"us_device_copy_cold_clean_l2": copy_us,
                      "frac_of_device_copy_cold": copy_us / cold_us})
        if it.mufu_ops:
            # two rooflines: HBM bytes and special-function unit operations
            # at the unit's rates measured in this run
            mufu_us = mufu_floor_us(it.mufu_ops, rates)
            hbm_us = it.bytes / (peak * 1e9) * 1e6
            d.update({"mufu_bound_us": mufu_us, "hbm_bound_us": hbm_us,
                      "bound": "mufu" if mufu_us > hbm_us else "hbm",
                      "frac_of_bound": max(mufu_us, hbm_us) / (ms * 1e3)})
            if pipe:
                d["frac_of_bound_in_pipeline"] = max(mufu_us, hbm_us) / pipe[it.name]
        per_chain[it.name] = d
    # next rows, measured beside the step (not part of its workload)
    next_rows = {}
    if args.only is None or re.search(args.only, f"layernorm_residual_{LN_ROWS[0]}x4096_bf16"):
        ln = _ln_item(dev, with_unfused=not args.no_unfused)
        st_us, st_per = steady_times(ln, 60)
        lms = st_us / 1e3
        ems = time_fn(ln.fused, reps=20, warm=3)
        cold_us = cold_time(ln, reps=20)
        d = {"bytes": ln.bytes, "us_fused": st_us, "gbs": ln.bytes / (lms / 1e3) / 1e9,
             "frac_of_" + peak_kind + "_peak": ln.bytes / (lms / 1e3) / 1e9 / peak,
             "us_events_one_launch": ems * 1e3,
             "frac_events_one_launch": ln.bytes / (ems / 1e3) / 1e9 / peak,
             "us_fused_cold_clean_l2": cold_us,
             "frac_cold_clean_l2": ln.bytes / (cold_us * 1e-6) / 1e9 / peak}
        if st_per:
            q = np.percentile(st_per, [10, 50, 90])
            d.update({"us_p10": q[0], "us_median": q[1], "us_p90": q[2]})
        if ln.unfused is not None:
            ums = time_fn(ln.unfused, reps=3, warm=1)
            d.update({"us_unfused": ums * 1e3, "unfused_kernels": ln.n_unfused,
                      "speedup": ums / lms})
        next_rows[ln.name] = d
        del ln
    if args.only is None or re.search(args.only, "rmsnorm_linear"):
        rl = _rms_linear_item(dev, with_unfused=not args.no_unfused, M=args.rl_m)
        tf_peak = tensor_peak()
        rms = time_fn(rl.fused, reps=10, warm=3)
        d = {"flops": rl.flops, "us_fused": rms * 1e3, "tflops": rl.flops / (rms / 1e3) / 1e12,
             "frac_of_bf16_peak": rl.flops / (rms / 1e3) / 1e12 / tf_peak[0],
             "bf16_peak_tflops": tf_peak[0], "peak_source": tf_peak[1],
             "us_gamma_per_call": time_fn(rl.gamma_path, reps=10, warm=3) * 1e3}
        if rl.unfused is not None:
            ums = time_fn(rl.unfused, reps=5, warm=2)
            d.update({"us_unfused": ums * 1e3, "unfused_kernels": rl.n_unfused,
                      "speedup": ums / rms})
            gms = time_fn(rl.library_gemm, reps=10, warm=3)
            d.update({"us_cublas_gemm_only": gms * 1e3, "fused_vs_cublas_gemm": gms / rms})
        next_rows[rl.name] = d
        del rl
    # rows beside the step that nothing else depends on: a failure is
    # reported in the line instead of ending the run
    extras = []
    if args.only is None or re.search(args.only, "rope_qkv_split_noalloc"):
        extras.append(("rope_qkv_split_noalloc", lambda: noalloc_row(dev, peak, peak_kind)))
    if args.only is None or re.search(args.only, "fast_math"):
        extras.append(("shuffle_chain_L16_fast_math", lambda: fast_math_row(
            dev, peak, peak_kind, rates)))
    for name, fn in extras:
        try:
            next_rows.update(fn())
        except Exception as e:
            next_rows[name] = {"error": str(e)[:300]}
    if (args.only is None or re.search(args.only, "decode_glue")) and not args.no_unfused:
        next_rows["decode_glue_32_layers_8_tokens"] = decode_glue(dev)
    # the chain sweep's smaller sizes (beside the step, not in it): 2^24 + 7
    # and 2^20 + 7 elements.  Cold: launches replayed from one graph, each on
    # the next of enough distinct buffer sets that together exceed twice the
    # L2, so every launch reads its inputs from HBM (the HBM fraction is taken
    # from this).  Warm: 20 launches on one buffer set replayed from a graph;
    # below L2 size that measures L2, not HBM, throughput, and no fraction of
    # the HBM peak is given for it.
    size_sweep = {}
    if args.only is None and args.spec is None and args.flat_elems is None:
        import workloads as W
        for n in (W.FLAT_SIZES[3], W.FLAT_SIZES[1]):
            for L in W.CHAIN_LENGTHS:
                spec, dt = W.random_chain(L, 5)
                c = F.fuse_compile(spec, (n,), dt)
                nb = sum(n * _esz(d) for d in c.in_dtypes) + n * _esz(c.out_dtype)
                nsets = int(2 * L2_BYTES // nb) + 2
                sets = []
                for k in range(nsets):
                    ins = [W.device_uniform(n, -2.0, 2.0, 300 + L * 7 + j + 1000 * k, d, dev)
                           for j, d in enumerate(c.in_dtypes)]
                    sets.append((ins, torch.empty(n, dtype=_tdt(c.out_dtype), device=dev)))
                ins, out = sets[0]
                warm_ms = graph_per_launch(lambda: F.fuse_launch(c, ins, out), k=20)
                reps = max(20, nsets)
                cyc = [0]

                def rotate():
                    i_s, o_s = sets[cyc[0] % nsets]
                    cyc[0] += 1
                    F.fuse_launch(c, i_s, o_s)
                cold_ms = graph_per_launch(rotate, k=reps - reps % nsets + nsets)
                d = {"bytes": nb, "us_fused": cold_ms * 1e3, "gbs": nb / (cold_ms / 1e3) / 1e9,
                     "frac_of_" + peak_kind + "_peak": nb / (cold_ms / 1e3) / 1e9 / peak,
                     "cold": f"{nsets} rotating buffer sets ({nsets * nb / 1e6:.0f} MB, over "
                             "twice the L2) replayed from one graph",
                     "us_fused_warm_graph": warm_ms * 1e3}
                if nb > L2_BYTES:
                    d["frac_warm_of_" + peak_kind + "_peak"] = nb / (warm_ms / 1e3) / 1e9 / peak
                else:
                    d["gbs_warm_l2_resident"] = nb / (warm_ms / 1e3) / 1e9
                size_sweep[f"flat_chain_L{L}_n{n}"] = d
                del sets, ins, out
    # dominant kernel and its roofline: its duration from the events around
    # it inside the timed region
    dit = items[dom]
    achieved = dit.bytes / (dom_ms / 1e3) / 1e9
    src_hash = kernel_source_hash(dit)
    traffic = traffic_record(dit.name, src_hash)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dit.name,
                "algorithmic_bytes": dit.bytes, "peak_source": peak_kind + " (burst copy)",
                "source_hash": src_hash, "us_per_launch": dom_ms * 1e3,
                "timing": "CUDA events around this kernel in every timed step"}
    # end to end: host (pinned) -> device copies of every input, the fused
    # launches, device -> host copies of every output, each step
    e2e = None
    if not args.no_e2e:
        max_in = max(t.numel() * t.element_size() for it in items for t in it.inputs)
        max_out = max(t.numel() * t.element_size() for it in items for t in it.outputs)
        # one pinned staging buffer holds the bytes of the largest input; each
        # input is copied from it (values do not change the timing)
        big = max((t for it in items for t in it.inputs), key=lambda t: t.numel() * t.element_size())
        h_in = torch.empty(max_in, dtype=torch.uint8, pin_memory=True)
        h_in.copy_(big.reshape(-1).view(torch.uint8))
        max_out = max(sum(t.numel() * t.element_size() for t in it.outputs) for it in items)
        h_out = torch.empty(max_out, dtype=torch.uint8, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for it in items for t in it.inputs)
        d2h = sum(t.numel() * t.element_size() for it in items for t in it.outputs)

        # three streams: host->device copies, kernels, device->host copies.
        # Item i's kernel waits for its inputs; its outputs are copied out
        # while later items compute; across steps, an item's inputs are not
        # overwritten before its previous kernel ran, and its outputs not
        # before they were copied out.
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        n_it = len(items)
        ev_in = [torch.cuda.Event() for _ in range(n_it)]
        ev_k = [torch.cuda.Event() for _ in range(n_it)]
        ev_out = [torch.cuda.Event() for _ in range(n_it)]
        first = [True]

        def e2e_step():
            for i, it in enumerate(items):
                if not first[0]:
                    s_in.wait_event(ev_k[i])
                with torch.cuda.stream(s_in):
                    for t in it.inputs:
                        nb = t.numel() * t.element_size()
                        t.view(-1).view(torch.uint8).copy_(h_in[:nb], non_blocking=True)
                ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if not first[0]:
                    stream.wait_event(ev_out[i])
                it.fused()
                ev_k[i].record(stream)
                s_out.wait_event(ev_k[i])
                with torch.cuda.stream(s_out):
                    off = 0
                    for t in it.outputs:
                        nb = t.numel() * t.element_size()
                        h_out[off:off + nb].copy_(t.view(-1).view(torch.uint8), non_blocking=True)
                        off += nb
                ev_out[i].record(s_out)
            first[0] = False
        e2e_steps = max(1, min(args.steps, 3))
        e2e_step()
        torch.cuda.synchronize()
        # the host side of the copies varies from second to second on a shared
        # node (115-182 ms for the same step, back to back): five timed runs
        # of e2e_steps steps each, the median reported, every run listed
        runs = []
        for _ in range(5):
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s_in.wait_event(a)
            for _ in range(e2e_steps):
                e2e_step()
            stream.wait_stream(s_out)
            b.record(stream)
            b.synchronize()
            runs.append(max_over_ranks(a.elapsed_time(b), world, dev) / e2e_steps)
        barrier()
        e_ms = statistics.median(runs)
        e2e = {"value": job_gbs(step_bytes, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": e2e_steps, "ms_per_step_runs": runs}
        # the host link bounds it: the step's copies cannot take less than
        # max(in / h2d rate, out / d2h rate).  The both-ways probe (equal bytes
        # each way) is reported but not used: when one direction is much
        # slower its time measures that direction, not a shared capacity
        link = link_rates(h_in, h_out, dev)
        bound = link_bound(step_bytes, world, h2d, d2h, link)
        e2e.update({"link_gbs": link, "link_bound": bound,
                    "frac_of_link_bound": e2e["value"] / bound})
    cpu = None
    if rank == 0 and not args.no_cpu:
        b, t, desc = cpu_sample(64)
        cpu = {"value": b / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": desc + f" ({sample_share(64)})", "seconds": t,
               "host_cores": os.cpu_count(), "nproc": len(os.sched_getaffinity(0))}
        ab, at, athreads, adesc = cpu_sample_all_cores(64)
        cpu["all_cores"] = {"value": ab / at / 1e9, "unit": UNIT, "cores": athreads,
                            "sample": adesc, "seconds": at}
    latency = None
    if rank == 0 and args.only is None and args.spec is None:
        import workloads as W
        spec, dt = W.random_chain(32, 5)
        try:
            latency = compile_latency(spec, W.FLAT_SIZES[-1], dt)
        except Exception as e:
            latency = {"error": str(e)[:300]}
    clk = clocks.summary()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2: each step streams "
                             f"{step_bytes / 1e9:.1f} GB, evicting the small workloads' buffers",
                       "storage_dtypes": "f32/f16/bf16 per workload, arithmetic in f32"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "per_chain": per_chain, "mufu_rates": mufu_report,
            "per_chain_timing": "us_fused (gbs, frac_of_*_peak): the workload on its own, 60 "
                                "launches (10 above 1 GB) back to back on rotating buffer sets "
                                "that together exceed twice the L2, replayed from one graph, mean "
                                "from events around the replay; us_p10/us_median/us_p90: the same "
                                "launches, end of each kernel minus the end of the one before "
                                "(CUPTI); us_in_step_events: the step's launches again with an "
                                "event between every two (each time includes the launch gap the "
                                f"event causes; that pass: {ms_per_step_item_events:.4f} ms a "
                                "step); us_in_pipeline: end of the workload's kernel minus end of "
                                "the one before, from the CUPTI trace of up to 20 undisturbed "
                                "steps" + (f" ({pipe_step_us / 1e3:.4f} ms a step)" if pipe else "")
                                + "; us_fused_cold_clean_l2: one launch after L2 is evicted with "
                                "clean lines, events around it, mean of 40 (5 above 1 GB)",
            "next_rows": next_rows, "size_sweep": size_sweep,
            "compile_cache": latency,
            "partial": ({"only": args.only, "flat_elems": args.flat_elems, "spec": args.spec}
                        if args.only or args.flat_elems or args.spec else None),
            "frac_of_peak": value / world / peak, "peak_gbs": peak}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def link_bound(step_bytes, world, h2d_bytes, d2h_bytes, link):
    """The most an end-to-end step can reach (GB/s of its algorithmic bytes)
    when its copies are the only limit: the inputs cannot arrive faster than
    the host-to-device rate nor the outputs leave faster than the
    device-to-host rate, each measured alone."""
    t_min = max(h2d_bytes / (link["h2d"] * 1e9), d2h_bytes / (link["d2h"] * 1e9))
    return job_gbs(step_bytes, world, t_min * 1e3)


def link_rates(h_in, h_out, dev, reps=4, rounds=5):
    """Host-link copy rates in GB/s, measured in the same run on the e2e
    pipeline's pinned buffers: host -> device alone, device -> host alone, and
    both at once on two streams (all bytes over the time).  The host side of
    these copies varies from second to second on a shared node, so each rate
    is the best of `rounds` measurements taken in turn with the others: the
    link's capacity, which is what a bound needs."""
    import torch
    nb = min(h_in.numel(), h_out.numel(), 512 << 20)
    d_in = torch.empty(nb, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nb, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(up, down):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s1)
        s2.wait_event(a)
        for _ in range(reps):
            if up:
                with torch.cuda.stream(s1):
                    d_in.copy_(h_in[:nb], non_blocking=True)
            if down:
                with torch.cuda.stream(s2):
                    h_out[:nb].copy_(d_out, non_blocking=True)
        s1.wait_stream(s2)
        b.record(s1)
        b.synchronize()
        return reps * nb * (int(up) + int(down)) / (a.elapsed_time(b) / 1e3) / 1e9

    timed(True, True)  # warm
    best = {"h2d": 0.0, "d2h": 0.0, "both": 0.0}
    for _ in range(rounds):
        best["h2d"] = max(best["h2d"], timed(True, False))
        best["d2h"] = max(best["d2h"], timed(False, True))
        best["both"] = max(best["both"], timed(True, True))
    rates = dict(best, bytes_per_copy=nb, rounds=rounds)
    del d_in, d_out
    return rates


def device_ops(fn):
    """The device activities (kernels, copies, memsets) of one call of fn, from
    CUPTI's records through torch.profiler: a list of (start_us, end_us, name)
    in start order."""
    import torch
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    ops = []
    for e in prof.profiler.kineto_results.events():
        if e.device_type() == torch.autograd.DeviceType.CUDA:
            t0 = e.start_ns() / 1e3
            ops.append((t0, t0 + e.duration_ns() / 1e3, e.name()))
    return sorted(ops)


def pipeline_times(items, steps):
    """Each workload's cost inside the back-to-back step, from the kernels'
    own end times: `steps` steps run under the CUPTI activity trace
    (torch.profiler), which timestamps every kernel without serialising the
    launches, and a workload's time is the end of its kernel minus the end of
    the kernel before it.  With programmatic dependent launch a kernel's CTAs
    may start before the previous kernel ends, so end-to-end differences, not
    start-to-end durations, are what each kernel adds.  Returns
    ({name: mean us}, mean step us), or (None, None) if the trace does not hold
    one kernel per workload per step."""
    import torch
    from torch.profiler import ProfilerActivity, profile
    device_ops(lambda: None)  # the process's first session can miss records
    n = len(items)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        for _ in range(steps):
            for it in items:
                it.fused()
        torch.cuda.synchronize()
    ends = sorted((e.start_ns() + e.duration_ns()) / 1e3 for e in prof.profiler.kineto_results.events()
                  if e.device_type() == torch.autograd.DeviceType.CUDA)
    if len(ends) != steps * n or steps < 2:
        return None, None
    per = {it.name: statistics.mean(ends[k * n + i] - ends[k * n + i - 1] for k in range(1, steps))
           for i, it in enumerate(items)}
    return per, (ends[-1] - ends[n - 1]) / (steps - 1)


def launch_trace(items):
    """Per workload, the fused launch against the unfused per-op sequence, as
    a timeline profiler shows them: device activities, their summed busy time,
    the span from the first start to the last end, and the idle gaps inside
    that span (span - busy), plus the time of the whole call measured with
    CUDA events outside the profiler."""
    import torch
    device_ops(lambda: None)  # the process's first session can miss records
    out = {}
    for it in items:
        rec = {}
        for mode, fn in (("fused", it.fused), ("unfused", it.unfused)):
            if fn is None:
                continue
            fn()  # warm: compiled, allocated, cached
            ops = device_ops(fn)
            if not ops:
                rec[mode] = {"device_ops": 0}
                continue
            busy = sum(b - a for a, b, _ in ops)
            span = ops[-1][1] - ops[0][0]
            names = {}
            for _, _, n in ops:
                k = n.split("<")[0].split("(")[0][:60]
                names[k] = names.get(k, 0) + 1
            rec[mode] = {"device_ops": len(ops), "busy_us": busy, "span_us": span,
                         "gaps_us": max(0.0, span - busy),
                         "us_events": time_fn(fn, reps=5, warm=1) * 1e3,
                         "ops_by_name": names}
        if "unfused" in rec:
            rec["declared_unfused_kernels"] = it.n_unfused
        out[it.name] = rec
    torch.cuda.synchronize()
    return out


def run_sequences_once(args, items, dev):
    """Each workload's fused call, then its unfused sequence, once each inside
    an NVTX range named "seq" (after an untimed warm-up of both), for a
    profiler that counts per-kernel DRAM bytes.  Profile it on the small case
    (--small: a few GB on the device), never at full size:
        ncu --nvtx --nvtx-include "seq/" --clock-control none \
            --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \
            python bench.py --sequences-once --small
    Prints the workloads in order with their unfused kernel counts, which
    attribute the profiler's kernel list to them."""
    import torch
    extra = []
    if args.only is None or re.search(args.only, f"layernorm_residual_{LN_ROWS[0]}x4096_bf16"):
        extra.append(_ln_item(dev, with_unfused=True))
    if args.only is None or re.search(args.only, "rmsnorm_linear"):
        extra.append(_rms_linear_item(dev, with_unfused=True, M=args.rl_m))
    order = []
    for it in items + extra:
        it.fused()
        if it.unfused is not None:
            it.unfused()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("seq")
        it.fused()
        if it.unfused is not None:
            it.unfused()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        order.append({"name": it.name, "bytes": it.bytes,
                      "unfused_kernels": it.n_unfused if it.unfused is not None else 0})
    print(json.dumps({"sequences": order}))
    return 0


def run_launch_trace(args, items, dev):
    extra = []
    if args.only is None or re.search(args.only, f"layernorm_residual_{LN_ROWS[0]}x4096_bf16"):
        extra.append(_ln_item(dev, with_unfused=True))
    if args.only is None or re.search(args.only, "rmsnorm_linear"):
        extra.append(_rms_linear_item(dev, with_unfused=True, M=args.rl_m))
    print(json.dumps({"launch_trace": launch_trace(items + extra)}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fused", choices=["fused", "reference"])
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", default=None, help="regex: run only the matching workloads")
    ap.add_argument("--flat-elems", type=int, default=None, help="size of the flat chains")
    ap.add_argument("--spec", default=None, help="time this one chain (flat) instead")
    ap.add_argument("--rl-m", type=int, default=16384, help="M of the RMSNorm -> Linear row")
    ap.add_argument("--spec-dtype", default="f32", choices=["f32", "f16", "bf16"])
    ap.add_argument("--launch-trace", action="store_true",
                    help="print device-op counts and gaps of fused vs unfused sequences instead")
    ap.add_argument("--small", action="store_true",
                    help="profiling captures: flat chains at 2^24+7, RMSNorm and LayerNorm "
                         "4096 rows, RoPE 8192 tokens, RMSNorm->Linear M=4096 (a few GB)")
    ap.add_argument("--sequences-once", action="store_true",
                    help="run each fused call and unfused sequence once in an NVTX range "
                         "'seq', for a profiler")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.small:
        import workloads as W
        if args.flat_elems is None:
            args.flat_elems = W.FLAT_SIZES[3]
        W.RMSNORM["rows"] = 4096
        W.ROPE["tokens"] = 8192
        LN_ROWS[0] = 4096
        args.rl_m = 4096
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
