"""Acceptance rules of the GPU parity tests.

The stated tolerances: fp32 outputs within 1e-6 relative, fp16 outputs within
2 ulp, bf16 outputs within 8e-3 relative, copies and index work bit-exact.
"Relative" is to the magnitude of the result's terms where a result is a sum
or difference of terms that can cancel (a rotation, x - mean, a dot product);
the oracle returns that magnitude beside the value.

Where a worst-case bound on the error of an fp32 evaluation is larger than the
flat tolerance, the bound is the tolerance, and it is derived here from the
kernel's arithmetic (each derivation is stated at its function):

* fp32 outputs pass when |g - ref| <= max(1e-6 * mag, E);
* fp16 outputs pass when g is within 2 ulp of the correctly rounded ref, or
  when g is a correct rounding of some value within E of ref (the device's
  fp32 result lies in [ref - E, ref + E] and the store rounds it);
* bf16 outputs pass when |g - ref| <= 8e-3 * mag.

Below the smallest normal number a correct rounding is off by up to half the
subnormal spacing in absolute terms, which no relative bound covers; that
much is added to the fp32 and bf16 rules (the fp16 rule counts ulps, which
already covers subnormals).

u = 2^-24 is the unit roundoff of fp32.  First-order bounds are multiplied by
1 + 1e-3, which covers their neglected higher-order terms many times over.
"""
import math

import numpy as np

import oracle

F32, F16, BF16 = oracle.F32, oracle.F16, oracle.BF16
U32 = 2.0 ** -24
SUB_HALF = {F16: 2.0 ** -25, BF16: 2.0 ** -134, F32: 2.0 ** -150}
HIGHER_ORDER = 1.0 + 1e-3


def f16_order(bits: np.ndarray) -> np.ndarray:
    """Monotone integer image of fp16 bit patterns (-0 and +0 both map to 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def accepted(got: np.ndarray, dt: int, ref: np.ndarray, mag=None, bound=None) -> np.ndarray:
    """Mask of device outputs that pass.

    got: device storage (float32 values, or uint16 bits for fp16/bf16);
    ref: the oracle's exact values; mag: magnitude of the terms (|ref| when
    None); bound: a derived bound E on |fp32 device value - ref| before the
    final store (0 when None).  Shapes broadcast against ref."""
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got).reshape(ref.shape)
    mag = np.abs(ref) if mag is None else np.broadcast_to(np.asarray(mag, np.float64), ref.shape)
    E = np.zeros_like(ref) if bound is None else np.broadcast_to(np.asarray(bound, np.float64),
                                                                 ref.shape)
    g = oracle.to_double(got, dt).reshape(ref.shape)
    with np.errstate(invalid="ignore"):
        if dt == F16:
            want = oracle.store(ref, F16)
            ok = np.abs(f16_order(got) - f16_order(want)) <= 2
            lo = f16_order(oracle.store(ref - E, F16))
            hi = f16_order(oracle.store(ref + E, F16))
            o = f16_order(got)
            ok |= (o >= lo) & (o <= hi)
        else:
            rel = 1e-6 if dt == F32 else 8e-3
            tol = np.maximum(rel * mag, E) if dt == F32 else rel * mag
            ok = np.abs(g - ref) <= tol + SUB_HALF[dt]
        nan = np.isnan(ref)
        ok = np.where(nan, np.isnan(g), ok)
        inf = np.isinf(ref)
        ok = np.where(inf, g == ref, ok)
    return ok


def assert_accepted(got, dt, ref, mag=None, bound=None, what=""):
    ok = accepted(got, dt, ref, mag, bound)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        g = oracle.to_double(np.asarray(got).reshape(np.shape(ref)), dt)
        r = np.asarray(ref).reshape(np.shape(g))
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; "
                             f"first at {bad.tolist()}: got {g[~ok][:5]}, want {r[~ok][:5]}")


# ------------------------------------------------------------ derived bounds

def reduction_depth(n: int) -> int:
    """Most fp32 additions any term of an n-term row sum passes through on the
    device: balanced trees per thread, over the lanes of a warp and over the
    warps of the CTA, each adding at most ceil(log2(nonzero terms)), so in all
    at most ceil(log2 n) + 3 (each of the three ceilings adds under one)."""
    return math.ceil(math.log2(max(n, 1))) + 3


def rmsnorm_rel_bound(hidden: int) -> float:
    """Relative error bound of an fp32 RMSNorm output y = h * rstd * w.

    h = x + res rounded (u); each square rounded once and summed through d
    additions ((d + 3) u on the sum, the squares of the rounded h included);
    the division by the row length and the add of eps (u each); the square
    root halves the relative error and rounds (u); the reciprocal (u):
    rstd is within (d + 9)/2 u.  Then h's own rounding and the two products
    (3 u): (d + 15)/2 u in all, d = reduction_depth(hidden).  It is below
    1e-6 up to rows of 2^15 and 1.013e-6 at 2^16."""
    d = reduction_depth(hidden)
    return HIGHER_ORDER * (d + 15) / 2 * U32


def layernorm_bound(h: np.ndarray, gamma, y: np.ndarray, eps: float) -> np.ndarray:
    """Bound E on |fp32 device LayerNorm output - exact value|, per element.

    h: exact h = x + residual, [rows, n]; gamma: the stored values as
    binary64 (None = absent); y: the exact outputs.  Two passes, each a
    tree of depth d = reduction_depth(n):
      mean: the tree, the division and h's own rounding leave
            delta_mu = (d + 2) u A from the exact mean, A = mean(|h|);
      var:  the deviations (h - mean) rounded, squared and summed:
            (d + 3) u; the division and eps: (d + 5) u; a mean off by
            delta_mu adds delta_mu^2; h's rounding moves the sum of squares
            by at most 2 u sqrt(M2 * sum h^2), i.e. 2 u q relative to
            V = var + eps with q = sqrt(mean(h^2) / V);
      rstd: rho = (d + 9)/2 u + q u + delta_mu^2 / (2 V);
      out:  (h - mean) off by u|h| + delta_mu + u|h - mean|, then rstd's
            rho and the products and the add (3 u):
      E = s |gamma| (u |h| + delta_mu + (rho + 3u)(|h| + A)) + u |y|,
    with s = 1/sqrt(V).  A derivation in the style of Higham, "Accuracy and
    Stability of Numerical Algorithms", chapters 3-4 (first order)."""
    h = np.asarray(h, np.float64)
    rows, n = h.shape
    d = reduction_depth(n)
    A = np.abs(h).mean(axis=1, keepdims=True)
    mu = h.mean(axis=1, keepdims=True)
    V = ((h - mu) ** 2).mean(axis=1, keepdims=True) + eps
    q = np.sqrt((h * h).mean(axis=1, keepdims=True) / V)
    dmu = (d + 2) * U32 * A
    rho = (d + 9) / 2 * U32 + q * U32 + dmu * dmu / (2 * V)
    s = 1.0 / np.sqrt(V)
    g = np.ones(n) if gamma is None else np.abs(np.asarray(gamma, np.float64))
    E = s * g * (U32 * np.abs(h) + dmu + (rho + 3 * U32) * (np.abs(h) + A)) + U32 * np.abs(y)
    return HIGHER_ORDER * E


def rope_bound(mag: np.ndarray, pair_abs: np.ndarray, positions) -> np.ndarray:
    """Bound E on |fp32 device RoPE output - exact value|.

    o = x1 cos - x2 sin: the cos/sin table is built in fp64 and rounded to
    fp32 (u on each term), one product and one fused multiply-add or
    subtraction round (2 u of the terms' magnitude at most): 3 u * mag.  The
    angle pos * base^(-2i/D) is formed in binary64 by both the table and the
    oracle (relative error a few 2^-53); its absolute error, up to
    pos * 2^-50, moves the output by at most that times |x1| + |x2|
    (pair_abs)."""
    pos = np.asarray(positions, np.float64).reshape(1, -1, 1)
    return HIGHER_ORDER * (3 * U32 * mag + pair_abs * pos * 2.0 ** -50)


def rope_pair_abs(qkv: np.ndarray, dt: int, heads: int, hd: int, which: int) -> np.ndarray:
    """|x1| + |x2| of the rotation pair behind every q (which 0) or k (1)
    output, as [heads, tokens, hd] binary64 (qkv: [tokens, 3*heads*hd]
    storage of dtype dt)."""
    T = qkv.shape[0]
    x = np.abs(oracle.to_double(qkv, dt).reshape(T, 3, heads, hd)[:, which])
    half = hd // 2
    p = x[..., :half] + x[..., half:]
    return np.concatenate([p, p], axis=-1).transpose(1, 0, 2)


def contraction_bound(mag: np.ndarray, dt: int, K: int, s_abs_x_scale: np.ndarray) -> np.ndarray:
    """Bound E on |device RMSNorm -> Linear output (before its store) - exact|.

    The product w * gamma is rounded once to the operand dtype (unit roundoff
    2^-11 for fp16, 2^-8 for bf16), and where it falls below the smallest
    normal the rounding is absolute, at most half the subnormal spacing
    (2^-25 for fp16) times |x| per term (s_abs_x_scale = |scale| * s *
    sum_k |x_k|).  The tensor cores accumulate in fp32 with at most one
    rounding, of up to an ulp (2u: they may truncate, as measured on earlier
    generations by Fasi, Higham, Mikaitis and Pranesh, "Numerical behavior
    of NVIDIA tensor cores", 2021), per k-step: 2 K u of the terms'
    magnitude; the row statistics, the scale and the bias add a few u more
    (32 u allowed)."""
    ud = 2.0 ** -11 if dt == F16 else 2.0 ** -8
    sub = 2.0 ** -25 if dt == F16 else 2.0 ** -134
    return HIGHER_ORDER * ((ud + (2 * K + 32) * U32) * mag + sub * s_abs_x_scale)
