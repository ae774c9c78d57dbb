"""Pins for the oracle's RMSNorm -> Linear -> scale ("TeleTron" section 4.2).

  * with an identity weight, scale 1 and no bias the result is the RMSNorm
    row (the separately pinned rmsnorm_residual with a zero residual);
  * bias and scale act affinely; the weight acts linearly;
  * scaling x leaves the result unchanged when eps = 0;
  * a one-hot row has a closed form;
  * evaluating a subset of rows gives those rows of the full result.
"""
import math

import numpy as np

import oracle
import workloads

BF = oracle.BF16


def _bf16(v):
    return oracle.store(np.asarray(v, np.float64), BF)


def _case(M=6, K=64, N=32, seed=0):
    x = workloads.normal((M, K), 0, 1, 500 + seed, BF)
    g = workloads.normal(K, 1, 0.1, 501 + seed, BF)
    w = workloads.normal((N, K), 0, 0.05, 502 + seed, BF)
    b = workloads.normal(N, 0, 0.1, 503 + seed, BF)
    return x, g, w, b


def test_identity_weight_gives_the_rmsnorm_row():
    M, K = 5, 64
    x = workloads.normal((M, K), 0, 1, 510, BF)
    g = workloads.normal(K, 1, 0.1, 511, BF)
    out, _ = oracle.rmsnorm_linear(x, g, _bf16(np.eye(K)), None, BF, 1e-6, 1.0)
    y, _ = oracle.rmsnorm_residual(x, _bf16(np.zeros((M, K))), g, BF, 1e-6)
    np.testing.assert_allclose(out, y, rtol=1e-12, atol=1e-14)


def test_bias_and_scale_are_affine_and_weight_is_linear():
    x, g, w, b = _case()
    base, _ = oracle.rmsnorm_linear(x, g, w, None, BF, 1e-6, 1.0)
    withb, _ = oracle.rmsnorm_linear(x, g, w, b, BF, 1e-6, 2.5)
    np.testing.assert_allclose(withb, 2.5 * (base + oracle.to_double(b, BF)), rtol=1e-12, atol=1e-12)
    wd = oracle.to_double(w, BF)
    w2 = _bf16(2 * wd)  # exact in bf16
    twice, _ = oracle.rmsnorm_linear(x, g, w2, None, BF, 1e-6, 1.0)
    np.testing.assert_allclose(twice, 2 * base, rtol=1e-12, atol=1e-14)


def test_scale_invariance_in_x():
    x, g, w, b = _case(seed=1)
    a, _ = oracle.rmsnorm_linear(x, g, w, b, BF, 0.0, 1.0)
    x4 = _bf16(4 * oracle.to_double(x, BF))
    a4, _ = oracle.rmsnorm_linear(x4, g, w, b, BF, 0.0, 1.0)
    np.testing.assert_allclose(a4, a, rtol=1e-12, atol=1e-12)


def test_one_hot_row_closed_form():
    K, N, eps, c, j = 64, 16, 1e-6, 3.0, 9
    x = np.zeros((1, K))
    x[0, j] = c
    _, g, w, b = _case(M=1, K=K, N=N, seed=2)
    out, _ = oracle.rmsnorm_linear(_bf16(x), g, w, b, BF, eps, 0.5)
    s = 1 / math.sqrt(c * c / K + float(np.float32(eps)))
    gd, wd, bd = (oracle.to_double(a, BF) for a in (g, w, b))
    want = 0.5 * (c * s * gd[j] * wd[:, j] + bd)
    np.testing.assert_allclose(out[0], want, rtol=1e-13)


def test_row_subset_matches_full():
    x, g, w, b = _case(M=9, seed=3)
    full, fm = oracle.rmsnorm_linear(x, g, w, b, BF, 1e-6, 1.0)
    sub, sm = oracle.rmsnorm_linear(x, g, w, b, BF, 1e-6, 1.0, rows=[7, 2])
    assert np.array_equal(sub, full[[7, 2]]) and np.array_equal(sm, fm[[7, 2]])
