"""Seeded synthetic inputs for the fused-chain workloads.

This module only draws random numbers and rounds them to a storage dtype; it
holds none of the method's arithmetic.  Both sides of every parity check (the
CUDA path and the oracle) receive the same stored values from here.

Storage conventions: fp32 -> numpy float32; fp16 and bf16 -> numpy uint16 bit
patterns (the raw 2-byte encodings).  Values are drawn in binary64 and rounded
to the storage dtype once (nearest-even).

The five workloads (sizes as the detection-head / transformer / ShuffleNet
layers they stand for):
  1. add -> relu -> scale: two fp32 vectors of 1,048,576, U[-1,1], scale 0.5
  2. detection-head decode: fp16 [1,255,80,80], [1,255,40,40], [1,255,20,20],
     N(0, sd 2), strides 8/16/32, three anchors per scale
  3. residual add + RMSNorm + cast: bf16 x, residual [16384, 4096] ~ N(0,1),
     weight 1 + 0.1 N(0,1), eps 1e-6
  4. QKV split + transpose + RoPE: bf16 qkv [32768, 3*32*128] ~ N(0,1),
     base 10000, positions 0..32767
  5. chain sweep: random chains of length 1..32 over {add, mul, sigmoid, exp,
     relu, scale, cast fp16<->fp32}, inputs U[-2,2]; (a) after a ChannelShuffle
     of 4 groups on fp16 [32,256,56,56]; (b) flat at 2^20, 2^24, 2^28 elements
     and each + 7
"""
from __future__ import annotations

import numpy as np

F32, F16, BF16 = 0, 1, 2

# ---------------------------------------------------------------- workloads

ADD_RELU_SCALE = dict(n=1 << 20, spec="add;relu;scale:0.5", lo=-1.0, hi=1.0, seed=1)

DETECT = dict(
    hw=[(80, 80), (40, 40), (20, 20)],
    strides=[8.0, 16.0, 32.0],
    na=3,
    no=85,
    sd=2.0,
    seed=2,
)

RMSNORM = dict(rows=16384, hidden=4096, eps=1e-6, seed=3)

ROPE = dict(tokens=32768, heads=32, head_dim=128, base=10000.0, pos0=0, seed=4)

SHUFFLE_CHAIN = dict(shape=(32, 256, 56, 56), groups=4, lo=-2.0, hi=2.0, seed=5)
FLAT_SIZES = [1 << 20, (1 << 20) + 7, 1 << 24, (1 << 24) + 7, 1 << 28, (1 << 28) + 7]
CHAIN_LENGTHS = [1, 2, 4, 8, 16, 32]


def detect_anchors(strides, na: int = 3) -> np.ndarray:
    """Fixed synthetic anchor boxes (the pages give none): for scale s and
    anchor a, (stride_s * 1.5 * (a + 1), stride_s * 2 * (a + 1)) pixels."""
    out = np.empty((len(strides), na, 2), np.float64)
    for s, st in enumerate(strides):
        for a in range(na):
            out[s, a] = (st * 1.5 * (a + 1), st * 2.0 * (a + 1))
    return out


# ---------------------------------------------------------------- rounding to storage

def _to_storage(x64: np.ndarray, dt: int) -> np.ndarray:
    if dt == F32:
        return x64.astype(np.float32)
    if dt == F16:
        return x64.astype(np.float16).view(np.uint16)
    # bf16: nearest-even from the float32 bit pattern (generation only; values
    # are first rounded to float32, which is fine for drawing random inputs)
    f = x64.astype(np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(shape, lo: float, hi: float, seed: int, dt: int) -> np.ndarray:
    x = rng(seed).uniform(lo, hi, size=shape)
    return _to_storage(x, dt)


def normal(shape, mean: float, sd: float, seed: int, dt: int) -> np.ndarray:
    x = rng(seed).normal(mean, sd, size=shape)
    return _to_storage(x, dt)


# ---------------------------------------------------------------- random chains

_OPS = ["add", "mul", "sigmoid", "exp", "relu", "scale", "cast"]


def random_chain(length: int, seed: int, start_dtype: int | None = None):
    """A random chain of `length` ops drawn uniformly from the sweep's op set.

    A cast switches the chain between fp16 and fp32.  Scale constants are
    multiples of 1/1024 in [0.5, 1.5], printed exactly, so that the literal is
    an fp32 value on both sides.  The start dtype is drawn from {fp16, fp32}
    unless given.  Returns (spec, start_dtype)."""
    g = rng(1_000_003 * length + seed)
    if start_dtype is None:
        start_dtype = F16 if int(g.integers(0, 2)) else F32
    cur = start_dtype
    items = []
    for _ in range(length):
        op = _OPS[int(g.integers(0, len(_OPS)))]
        if op == "scale":
            k = int(g.integers(512, 1537))
            items.append(f"scale:{k / 1024!r}")
        elif op == "cast":
            cur = F32 if cur == F16 else F16
            items.append("cast:" + ("f32" if cur == F32 else "f16"))
        else:
            items.append(op)
    return ";".join(items), start_dtype


def chain_inputs(spec: str, in_dtype: int, numel: int, seed: int, lo=-2.0, hi=2.0):
    """Storage arrays for every input of a chain: input 0 in in_dtype, then one
    tensor per add/mul in the chain's dtype at that op."""
    dts = [in_dtype]
    cur = in_dtype
    for item in (s.strip() for s in spec.split(";") if s.strip()):
        name, _, arg = item.partition(":")
        if name == "cast":
            cur = {"f32": F32, "f16": F16, "bf16": BF16}[arg]
        elif name in ("add", "mul"):
            dts.append(cur)
    return [uniform(numel, lo, hi, seed * 7919 + j, dt) for j, dt in enumerate(dts)], dts


# ---------------------------------------------------------------- device-side generation

def device_uniform(numel: int, lo: float, hi: float, seed: int, dt: int, device="cuda"):
    """Seeded uniform draw made on the GPU (for inputs too large to draw on the
    host quickly).  Returns a torch tensor of the storage dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.rand(numel, generator=g, device=device, dtype=torch.float32)
    x = x * (hi - lo) + lo
    return x.to({F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dt])


def device_normal(shape, mean: float, sd: float, seed: int, dt: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sd + mean
    return x.to({F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dt])
