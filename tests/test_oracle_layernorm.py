"""Pins for the oracle's residual add + LayerNorm (CPU only).

"DeepJIT" section 4.3: per row mean, variance as E[x^2] - mean^2, then
(x - mean) * rsqrt(var + eps) * gamma + beta; here with x + residual.  The
pins are properties fixed by the mathematics: unit gamma and zero beta give
rows of mean 0 and variance var/(var + eps); the affine parameters act
elementwise; a constant shift of the input changes nothing; a constant row
gives beta; a two-valued row has a closed form; the residual is summed
exactly.
"""
import numpy as np

import oracle
import workloads

BF = oracle.BF16


def _bf16(v):
    return oracle.store(np.asarray(v, np.float64), BF)


def test_unit_affine_rows_are_standardised():
    rows, hidden, eps = 32, 4096, 1e-6
    x = workloads.normal((rows, hidden), 0, 1, 71, BF)
    r = workloads.normal((rows, hidden), 0, 1, 72, BF)
    y, h, _ = oracle.layernorm_residual(x, r, None, None, BF, eps)
    var = h.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), var / (var + np.float32(eps)), rtol=1e-10)
    assert np.all(np.abs(y.var(axis=1) - 1) < 1e-6)


def test_gamma_beta_act_elementwise():
    rows, hidden = 8, 512
    x = workloads.normal((rows, hidden), 0, 1, 73, BF)
    g = workloads.normal(hidden, 1, 0.2, 74, BF)
    b = workloads.normal(hidden, 0, 0.5, 75, BF)
    y0, _, _ = oracle.layernorm_residual(x, None, None, None, BF, 1e-6)
    y, _, _ = oracle.layernorm_residual(x, None, g, b, BF, 1e-6)
    gd, bd = oracle.to_double(g, BF), oracle.to_double(b, BF)
    np.testing.assert_allclose(y, y0 * gd + bd, rtol=1e-12, atol=1e-12)


def test_shift_invariance_and_exact_residual():
    g = np.random.default_rng(76)
    a = g.integers(-50, 50, (6, 128)).astype(np.float64)
    b = g.integers(-50, 50, (6, 128)).astype(np.float64)
    y, h, _ = oracle.layernorm_residual(_bf16(a), _bf16(b), None, None, BF, 1e-6)
    assert np.array_equal(h, a + b)
    y2, _, _ = oracle.layernorm_residual(_bf16(a + 64), _bf16(b), None, None, BF, 1e-6)
    np.testing.assert_allclose(y2, y, rtol=1e-10, atol=1e-10)


def test_constant_row_gives_beta():
    x = _bf16(np.full((3, 64), 2.5))
    b = workloads.normal(64, 0, 1, 77, BF)
    y, _, _ = oracle.layernorm_residual(x, None, None, b, BF, 1e-6)
    assert np.array_equal(y, np.broadcast_to(oracle.to_double(b, BF), y.shape))


def test_two_valued_row_closed_form():
    # a row of +a and -a (mean 0, variance a^2): y = +-a / sqrt(a^2 + eps)
    eps = 1e-6
    for a in (1.0, 0.001, 3.0):
        row = np.tile([a, -a], 32)
        ab = oracle.to_double(_bf16([a]), BF)[0]
        y, _, _ = oracle.layernorm_residual(_bf16(row[None, :]), None, None, None, BF, eps)
        want = np.tile([ab, -ab], 32) / np.sqrt(ab * ab + np.float32(eps))
        np.testing.assert_allclose(y[0], want, rtol=1e-12)


def test_term_magnitudes_by_hand():
    # row h = (-1, 3): mean 1, mean(|h|) 2, var 4; eps 0 gives s = 1/2.
    # y = (h - mean) s gamma + beta has the terms h s gamma, -mean s gamma
    # and beta, and the mean is the sum of the terms h_k / 2, whose
    # magnitudes add up to mean(|h|) = 2 (not |mean| = 1):
    #   mag_k = (|h_k| + 2) * s * |gamma_k| + |beta_k|
    x = _bf16([[-1.0, 3.0]])
    g = _bf16([2.0, -1.0])
    b = _bf16([0.5, -0.25])
    y, _, mag = oracle.layernorm_residual(x, None, g, b, BF, 0.0)
    assert y.tolist() == [[(-1 - 1) * 0.5 * 2 + 0.5, (3 - 1) * 0.5 * -1 - 0.25]]
    assert mag.tolist() == [[(1 + 2) * 0.5 * 2 + 0.5, (3 + 2) * 0.5 * 1 + 0.25]]
