"""Fuzzing the chain-spec parser (no GPU).

  * random strings never crash the library: fuse_source returns a source or
    a FUSE_E_SPEC / FUSE_E_SHAPE / FUSE_E_DTYPE error;
  * on random token sequences the library's parser and the oracle's own,
    independent parser agree on which specs are valid and, for the valid
    ones, on the number of inputs, every input's dtype and the output dtype
    (read from the generated source);
  * a sample of the valid random chains compiles with NVRTC.
"""
import random
import re

import numpy as np
import pytest

import elementwise_chain_jit_gb300 as F
import oracle

ALPHABET = "addmulscalerelusigmoidexpcastshuffle:;0123456789.-e f16bf32 \t"
VALID = ["add", "mul", "relu", "sigmoid", "exp", "scale:0.5", "scale:-1.25", "scale:3e-2",
         "cast:f16", "cast:bf16", "cast:f32"]
INVALID = ["cast:f64", "scale:x", "scale:", "foo", "reluu", "shuffle:2", "cast:", "scale:inf",
           "scale:nan", "scale:1e39", "relu:1", "add:2", "exp:", "shuffle:0", "shuffle:x"]
DTS = [F.F32, F.F16, F.BF16]


def _library(spec, shape, dt):
    """(None, error code) or ((n_in, in_dtypes, out_dtype), None) from the
    library's generated source."""
    try:
        src = F.fuse_source(spec, shape, dt)
    except F.FuseError as e:
        return None, e.code
    n_in = int(re.search(r"constexpr int NIN = (\d+);", src).group(1))
    dts = [int(re.search(rf"constexpr int DT{j} = (\d+);", src).group(1)) for j in range(n_in)]
    out = int(re.search(r"constexpr int DTO = (\d+);", src).group(1))
    return (n_in, dts, out), None


def _oracle(spec, dt, shape):
    try:
        ch = oracle.parse_spec(spec, dt)
    except (ValueError, KeyError):
        return None
    # the shape rule of a shuffle: NCHW with C divisible by the groups
    if ch.groups and (len(shape) != 4 or shape[1] % ch.groups):
        return None
    return len(ch.in_dtypes), list(ch.in_dtypes), ch.out_dtype


def test_random_strings_never_crash():
    rng = random.Random(1)
    for _ in range(3000):
        spec = "".join(rng.choice(ALPHABET) for _ in range(rng.randint(0, 40)))
        info, code = _library(spec, (37,), rng.choice(DTS))
        assert info is not None or code in (-1, -2, -3), (spec, code)


def test_library_and_oracle_parsers_agree():
    rng = random.Random(2)
    checked = valid = 0
    for _ in range(3000):
        items = [rng.choice(VALID if rng.random() < 0.9 else INVALID)
                 for _ in range(rng.randint(0, 12))]
        shuffle = rng.random() < 0.3
        if shuffle:
            items = [f"shuffle:{rng.choice([1, 2, 3, 4, 6, 12])}"] + items
            shape = (2, 12, 3, 5)
        else:
            shape = (257,)
        if rng.random() < 0.2:  # stray separators and spaces
            items = [f" {s} " for s in items] + [""]
        spec = ";".join(items)
        dt = rng.choice(DTS)
        lib, code = _library(spec, shape, dt)
        ref = _oracle(spec, dt, shape)
        assert (lib is None) == (ref is None), (spec, lib, code, ref)
        if lib is not None:
            assert lib == ref, (spec, lib, ref)
            valid += 1
        checked += 1
    assert valid > 1000 and checked == 3000


@pytest.mark.parametrize("seed", range(4))
def test_random_valid_chains_compile(seed):
    rng = random.Random(100 + seed)
    for _ in range(10):
        spec = ";".join(rng.choice(VALID) for _ in range(rng.randint(1, 16)))
        dt = rng.choice(DTS)
        c = F.fuse_compile(spec, (rng.randint(1, 5000),), dt)
        assert c.n_in == 1 + sum(s in ("add", "mul") for s in spec.split(";"))


def test_scale_literal_is_the_nearest_fp32_on_both_sides():
    # just above the midpoint of 1 and 1 + 2^-23: a literal rounded to
    # binary64 first lands on the midpoint and then ties down to 1; the
    # nearest fp32 is 1 + 2^-23
    lit = "1.000000059604644775390625000000000000001"
    assert oracle.parse_spec(f"scale:{lit}", F.F32).args[0] == 1 + 2 ** -23
    assert "x * 0x1.000002p+0f;" in F.fuse_source(f"scale:{lit}", (7,), F.F32)
    # the exact midpoint ties to the even neighbour, 1
    mid = "1.000000059604644775390625"
    assert oracle.parse_spec(f"scale:{mid}", F.F32).args[0] == 1.0
    assert "x * 0x1p+0f;" in F.fuse_source(f"scale:{mid}", (7,), F.F32)
    # the largest fp32 and just past its rounding range
    assert oracle.parse_spec("scale:3.4028235e38", F.F32).args[0] == float(np.finfo(np.float32).max)
    with pytest.raises(ValueError):
        oracle.parse_spec("scale:3.5e38", F.F32)
    with pytest.raises(F.FuseError):
        F.fuse_source("scale:3.5e38", (7,), F.F32)
