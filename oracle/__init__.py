"""Plain fp64 CPU oracle for the fused-chain hot path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  The product library never loads it, and it imports
nothing from the product: it has its own spec parser (below), its own dtype
conversions and its own arithmetic (``oracle.c``).

What each function follows is cited in ``oracle.c``.  The spec language read
here is the one the library's ``fuse_compile`` accepts::

    [shuffle:G;]op;op;...     op = add | mul | scale:<c> | relu | sigmoid
                                   | exp | sigmoid:fast | exp:fast
                                   | cast:f16 | cast:f32 | cast:bf16

``exp:fast`` and ``sigmoid:fast`` have the same exact value as exp and
sigmoid; only the error bound the check allows the device differs.

Reading of the multi-input chain of "DeepJIT" section 4.1 ((a + b) -> relu ->
scale -> + c): ``add`` and ``mul`` each consume the next input tensor, which
has the chain's current dtype; ``scale`` multiplies by an fp32 constant.
"""
from __future__ import annotations

import ctypes
import math
import os
import struct
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}
DTYPE_NAMES = {v: k for k, v in DTYPE_CODES.items()}
STORAGE = {F32: np.float32, F16: np.uint16, BF16: np.uint16}

OP_ADD, OP_MUL, OP_SCALE, OP_RELU, OP_SIGMOID, OP_EXP, OP_CAST = 1, 2, 3, 4, 5, 6, 7
OP_EXP_FAST, OP_SIGMOID_FAST = 8, 9
_UNARY = {"relu": OP_RELU, "sigmoid": OP_SIGMOID, "exp": OP_EXP}
_FAST = {"sigmoid": OP_SIGMOID_FAST, "exp": OP_EXP_FAST}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
                               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB names another build of oracle.c to load instead (the
        # mutation test points it at copies with a mistake planted)
        path = os.environ.get("ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        P, I64, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_round_f16.restype = D
        L.oracle_round_f16.argtypes = [D]
        L.oracle_round_bf16.restype = D
        L.oracle_round_bf16.argtypes = [D]
        L.oracle_round_f32.restype = D
        L.oracle_round_f32.argtypes = [D]
        L.oracle_store.argtypes = [P, I64, I, P]
        L.oracle_load.argtypes = [P, I, I64, P]
        L.oracle_chain_eval.argtypes = [I, P, P, P, P, P, I64, P, I, P, P]
        L.oracle_chain_check.restype = I64
        L.oracle_chain_check.argtypes = [I, P, P, P, P, P, I64, P, I, P, P, I, P, P]
        L.oracle_channel_shuffle.argtypes = [P, P, I64, I64, I64, I64, I, I]
        L.oracle_rmsnorm_residual.argtypes = [P, P, P, I, I64, I64, ctypes.c_float, P, P]
        L.oracle_rope_qkv_split.argtypes = [P, I, I64, I, I, P, D, P, P, P, P, P]
        L.oracle_layernorm_residual.argtypes = [P, P, P, P, I, I64, I64, ctypes.c_float, P, P, P]
        L.oracle_rmsnorm_linear.argtypes = [P, P, P, P, I, I64, I64, P, I64, ctypes.c_float,
                                            ctypes.c_float, P, P]
        L.oracle_detect_decode.argtypes = [P, I, P, P, P, I, I, I, P, P]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- dtypes

def to_double(raw: np.ndarray, dt: int) -> np.ndarray:
    """Exact binary64 value of stored elements (fp32 array, or uint16 bits)."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, np.float64)
    lib().oracle_load(_p(raw), dt, raw.size, _p(out))
    return out.reshape(raw.shape)


def store(values: np.ndarray, dt: int) -> np.ndarray:
    """Round binary64 values to dtype dt (nearest-even) and return the storage."""
    v = _c(values, np.float64)
    out = np.empty(v.size, STORAGE[dt])
    lib().oracle_store(_p(v), v.size, dt, _p(out))
    return out.reshape(v.shape)


def round_f16(x: float) -> float:
    return lib().oracle_round_f16(float(x))


def round_bf16(x: float) -> float:
    return lib().oracle_round_bf16(float(x))


def round_f32(x: float) -> float:
    return lib().oracle_round_f32(float(x))


# ---------------------------------------------------------------- chains

@dataclass
class Chain:
    ops: list            # op codes
    args: list           # scale constant (fp32 value) or cast target dtype
    in_idx: list         # input consumed by add/mul (else 0)
    in_dtypes: list      # dtype of every input tensor, input 0 first
    out_dtype: int
    groups: int          # ChannelShuffle groups on input 0 (0 = none)


def _f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def _f32_of_literal(text: str) -> float:
    """The fp32 value nearest the decimal literal's exact value, ties to even
    (a literal rounded to binary64 first can land on an fp32 midpoint and
    then round the wrong way).  Infinity beyond the fp32 range."""
    from fractions import Fraction
    exact = Fraction(text)
    try:
        c = _f32(float(exact))
    except OverflowError:
        return math.copysign(math.inf, exact)
    best = c
    with np.errstate(over="ignore"):
        neighbours = (np.nextafter(np.float32(c), np.float32(-np.inf)),
                      np.nextafter(np.float32(c), np.float32(np.inf)))
    for cand in neighbours:
        cand = float(cand)
        if not math.isfinite(cand):
            continue
        d_best, d_cand = abs(Fraction(best) - exact), abs(Fraction(cand) - exact)
        if d_cand < d_best or (d_cand == d_best and
                               struct.unpack("<I", struct.pack("<f", cand))[0] % 2 == 0):
            best = cand
    return best


def parse_spec(spec: str, in_dtype: int) -> Chain:
    """Read a spec into op codes, following the dtype through the casts."""
    ops, args, in_idx, in_dtypes = [], [], [], [in_dtype]
    groups, cur = 0, in_dtype
    items = [s.strip() for s in spec.split(";") if s.strip()]
    for pos, item in enumerate(items):
        name, colon, arg = item.partition(":")
        name, arg = name.strip(), arg.strip()
        if name == "shuffle":
            if pos != 0:
                raise ValueError("shuffle must come first")
            groups = int(arg)
            if not 0 < groups <= 1 << 20:
                raise ValueError("shuffle groups outside 1..2^20")
            continue
        fast = colon and name in _FAST and arg == "fast"
        if colon and name not in ("scale", "cast") and not fast:
            raise ValueError(f"{name!r} takes no argument (exp and sigmoid take 'fast')")
        if name in ("add", "mul"):
            ops.append(OP_ADD if name == "add" else OP_MUL)
            args.append(0.0)
            in_idx.append(len(in_dtypes))
            in_dtypes.append(cur)
        elif name == "scale":
            c = _f32_of_literal(arg)
            if not np.isfinite(c):
                raise ValueError("the scale constant must be finite in fp32")
            ops.append(OP_SCALE)
            args.append(c)
            in_idx.append(0)
        elif name in _UNARY:
            ops.append(_FAST[name] if fast else _UNARY[name])
            args.append(0.0)
            in_idx.append(0)
        elif name == "cast":
            cur = DTYPE_CODES[arg]
            ops.append(OP_CAST)
            args.append(float(cur))
            in_idx.append(0)
        else:
            raise ValueError(f"unknown op {item!r}")
    return Chain(ops, args, in_idx, in_dtypes, cur, groups)


def _chain_arrays(ch: Chain, inputs, shape):
    ins = [np.ascontiguousarray(a) for a in inputs]
    if len(ins) != len(ch.in_dtypes):
        raise ValueError(f"chain takes {len(ch.in_dtypes)} inputs, got {len(ins)}")
    ptrs = (ctypes.c_void_p * len(ins))(*[a.ctypes.data for a in ins])
    ops = np.array(ch.ops or [0], np.int32)
    args = np.array(ch.args or [0.0], np.float64)
    idx = np.array(ch.in_idx or [0], np.int32)
    dts = np.array(ch.in_dtypes, np.int32)
    nchw = np.array(list(shape) if ch.groups else [1, 1, 1, 1], np.int64)
    return ins, ptrs, ops, args, idx, dts, nchw


def chain_eval(spec: str, in_dtype: int, inputs, shape, idx=None):
    """Exact value (binary64) of each output element, before the final store.

    inputs: storage arrays (input 0 first); shape: the tensor shape (NCHW when
    the spec starts with shuffle); idx: optional output indices to evaluate.
    Returns (values, out_dtype)."""
    ch = parse_spec(spec, in_dtype)
    ins, ptrs, ops, args, iidx, dts, nchw = _chain_arrays(ch, inputs, shape)
    n = int(np.prod(shape)) if idx is None else len(idx)
    sel = None if idx is None else _c(idx, np.int64)
    out = np.empty(n, np.float64)
    lib().oracle_chain_eval(len(ch.ops), _p(ops), _p(args), _p(iidx), ptrs, _p(dts), n,
                            _p(sel), ch.groups, _p(nchw), _p(out))
    return out, ch.out_dtype


def chain_check(spec: str, in_dtype: int, inputs, shape, device_out, idx=None):
    """Classify device results: returns (fails, counts[4], classes).

    classes: 0 flat tolerance, 1 running error bound, 2 fail, 3 unpinned."""
    ch = parse_spec(spec, in_dtype)
    ins, ptrs, ops, args, iidx, dts, nchw = _chain_arrays(ch, inputs, shape)
    dev = np.ascontiguousarray(device_out).reshape(-1)
    if dev.dtype != STORAGE[ch.out_dtype]:
        raise ValueError("device output storage does not match the chain's output dtype")
    n = dev.size
    sel = None if idx is None else _c(idx, np.int64)
    cls = np.empty(n, np.int8)
    counts = np.zeros(4, np.int64)
    fails = lib().oracle_chain_check(len(ch.ops), _p(ops), _p(args), _p(iidx), ptrs, _p(dts), n,
                                     _p(sel), ch.groups, _p(nchw), _p(dev), ch.out_dtype,
                                     _p(cls), _p(counts))
    return int(fails), counts, cls


# ---------------------------------------------------------------- fixed ops

def channel_shuffle(x: np.ndarray, groups: int) -> np.ndarray:
    """ChannelShuffle of an NCHW array, element bytes copied unchanged."""
    x = np.ascontiguousarray(x)
    n, c, h, w = x.shape
    if c % groups:
        raise ValueError("channels must divide by groups")
    out = np.empty_like(x)
    lib().oracle_channel_shuffle(_p(x), _p(out), n, c, h, w, groups, x.itemsize)
    return out


def rmsnorm_residual(x, res, w, dt: int, eps: float):
    """Returns (y, residual_out) in binary64, shaped like x."""
    x, res, w = (np.ascontiguousarray(a) for a in (x, res, w))
    rows, hidden = x.shape
    y = np.empty((rows, hidden), np.float64)
    r = np.empty((rows, hidden), np.float64)
    lib().oracle_rmsnorm_residual(_p(x), _p(res), _p(w), dt, rows, hidden, ctypes.c_float(eps),
                                  _p(y), _p(r))
    return y, r


def rmsnorm_linear(x, gamma, w, bias, dt: int, eps: float, scale: float, rows=None):
    """scale * (RMSNorm(x) * gamma @ w.T + bias) for the given rows of x
    [M, K] (all rows if None); w is [N, K]; bias may be None.  Returns
    (out, term magnitudes), both [len(rows), N] in binary64."""
    x, gamma, w = (np.ascontiguousarray(a) for a in (x, gamma, w))
    bias = None if bias is None else np.ascontiguousarray(bias)
    M, K = x.shape
    N = w.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    out = np.empty((len(rows), N), np.float64)
    mag = np.empty((len(rows), N), np.float64)
    lib().oracle_rmsnorm_linear(_p(x), _p(gamma), _p(w), _p(bias), dt, K, N, _p(rows), len(rows),
                                ctypes.c_float(eps), ctypes.c_float(scale), _p(out), _p(mag))
    return out, mag


def layernorm_residual(x, res, gamma, beta, dt: int, eps: float):
    """LayerNorm of h = x + res (res, gamma, beta may be None).  Returns
    (y, residual_out or None, term magnitudes) in binary64, shaped like x."""
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    res, gamma, beta = (None if a is None else np.ascontiguousarray(a) for a in (res, gamma, beta))
    y = np.empty((rows, hidden), np.float64)
    mag = np.empty((rows, hidden), np.float64)
    ro = np.empty((rows, hidden), np.float64) if res is not None else None
    lib().oracle_layernorm_residual(_p(x), _p(res), _p(gamma), _p(beta), dt, rows, hidden,
                                    ctypes.c_float(eps), _p(y), _p(ro), _p(mag))
    return y, ro, mag


def rope_qkv_split(qkv, dt: int, heads: int, head_dim: int, positions, base: float = 10000.0):
    """qkv: [tokens, 3*heads*head_dim] storage.  Returns q, k, v, q_mag, k_mag
    as binary64 arrays shaped [heads, tokens, head_dim]."""
    qkv = np.ascontiguousarray(qkv)
    tokens = qkv.shape[0]
    pos = _c(positions, np.int64)
    shp = (heads, tokens, head_dim)
    q, k, v, qm, km = (np.empty(shp, np.float64) for _ in range(5))
    lib().oracle_rope_qkv_split(_p(qkv), dt, tokens, heads, head_dim, _p(pos), float(base),
                                _p(q), _p(k), _p(v), _p(qm), _p(km))
    return q, k, v, qm, km


def detect_decode(feats, dt: int, strides, anchors, na: int, no: int):
    """feats: list of [1, na*no, H, W] storage arrays.  anchors: [nscales, na, 2].
    Returns (out [rows, no], term_mag [rows, no]) in binary64."""
    feats = [np.ascontiguousarray(f) for f in feats]
    hw = np.array([d for f in feats for d in f.shape[2:]], np.int32)
    rows = sum(na * f.shape[2] * f.shape[3] for f in feats)
    ptrs = (ctypes.c_void_p * len(feats))(*[f.ctypes.data for f in feats])
    st = _c(strides, np.float64)
    an = _c(anchors, np.float64).reshape(-1)
    out = np.empty((rows, no), np.float64)
    mag = np.empty((rows, no), np.float64)
    lib().oracle_detect_decode(ptrs, dt, _p(hw), _p(st), _p(an), len(feats), na, no, _p(out),
                               _p(mag))
    return out, mag
