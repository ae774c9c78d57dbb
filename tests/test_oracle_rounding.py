"""Pins for the oracle's dtype conversions and rounding (CPU only).

The oracle converts stored fp16/bf16/fp32 values to binary64 and rounds to
nearest-even with its own code.  These tests hold it against independent
routines (numpy's float16/float32 casts, torch's bfloat16) and against
hand-derived ties and overflow cases.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(tok: str) -> float:
    tok = tok.strip()
    if tok.lower() in ("inf", "+inf", "-inf", "nan"):
        return float(tok)
    if "0x" in tok:
        return float.fromhex(tok)
    return float(tok)


def test_golden_rounding_cases():
    rows = 0
    for line in open(os.path.join(GOLDEN, "float_rounding.txt")):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        fmt, x, want = line.split()
        got = (oracle.round_f16 if fmt == "f16" else oracle.round_bf16)(_num(x))
        w = _num(want)
        assert got == w and np.signbit(got) == np.signbit(w), (fmt, x, got, w)
        rows += 1
    assert rows >= 10


def _doubles(seed, n=200_000):
    g = np.random.default_rng(seed)
    mant = g.uniform(1.0, 2.0, n)
    exp = g.integers(-30, 18, n)
    sign = np.where(g.random(n) < 0.5, -1.0, 1.0)
    x = sign * np.ldexp(mant, exp)
    return x


def _f16_ties():
    # exact midpoints between neighbouring fp16 values, and nudges around them
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = h.view(np.float16).astype(np.float64)
    b = (h + 1).view(np.float16).astype(np.float64)
    mid = (a + b) / 2
    return np.concatenate([mid, -mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)])


def test_round_f16_matches_numpy():
    x = np.concatenate([_doubles(1), _f16_ties(), [65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0]])
    got = oracle.to_double(oracle.store(x, oracle.F16), oracle.F16)
    with np.errstate(over="ignore"):  # values past the fp16 range round to inf, as intended
        want = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_round_f32_matches_numpy():
    g = np.random.default_rng(2)
    x = np.concatenate([_doubles(3) * 2.0 ** g.integers(-100, 100, 200_000),
                        [3.4028235677973366e38, 3.4028235677973362e38, 1e-46, -1e-45]])
    # exact midpoints between neighbouring fp32 values
    f = g.uniform(-1e3, 1e3, 50_000).astype(np.float32)
    up = np.nextafter(f, np.float32(np.inf))
    x = np.concatenate([x, (f.astype(np.float64) + up.astype(np.float64)) / 2])
    got = oracle.to_double(oracle.store(x, oracle.F32), oracle.F32)
    with np.errstate(over="ignore"):  # values past the fp32 range round to inf, as intended
        want = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest-even; on fp32-representable inputs
    # that is the direct rounding the oracle does from binary64
    g = np.random.default_rng(4)
    f = (g.standard_normal(300_000) * 2.0 ** g.integers(-60, 60, 300_000)).astype(np.float32)
    bits = np.arange(0, 0x7F7F, 7, dtype=np.uint32) << 16
    ties = (bits | 0x8000).view(np.float32)  # exact bf16 midpoints
    f = np.concatenate([f, ties, -ties])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.store(f.astype(np.float64), oracle.BF16)
    assert np.array_equal(got, want)


def test_load_all_fp16_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.to_double(h, oracle.F16)
    want = h.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_load_all_bf16_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.to_double(h, oracle.BF16)
    want = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("dt", [oracle.F16, oracle.BF16])
def test_store_load_round_trip(dt):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.to_double(h, dt)
    keep = ~np.isnan(v)
    assert np.array_equal(oracle.store(v[keep], dt), h[keep])
