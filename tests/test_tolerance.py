"""CPU checks of the GPU tests' acceptance rules (tests/tolerance.py): they
accept what the stated tolerances accept and refuse what they refuse, and the
derived bounds hold for an fp32 evaluation simulated with numpy in the
kernels' order of operations (balanced trees, fp32 roundings)."""
import numpy as np

import oracle
import tolerance as tol
import workloads

F32, F16, BF16 = oracle.F32, oracle.F16, oracle.BF16


def _f16_bits(v):
    return np.asarray(v, np.float16).view(np.uint16)


def test_f16_rule_counts_ulps():
    ref = np.array([1.0, 1.0, 1.0, 6.0e-8, -2.0])
    ulp = 2.0 ** -10
    got = _f16_bits([1.0 + 2 * ulp, 1.0 - 2 * ulp / 2, 1.0 + 3 * ulp, 3 * 2.0 ** -24, -2.0])
    ok = tol.accepted(got, F16, ref)
    assert ok.tolist() == [True, True, False, True, True]
    # a bound E wide enough to reach the third value accepts it
    assert tol.accepted(got[2:3], F16, ref[2:3], bound=3.0 * ulp).all()


def test_fp32_and_bf16_rules():
    # the last two: below the smallest normal, a correct rounding of 0.6 of
    # the subnormal spacing is one spacing (accepted); two spacings are not
    sub = 2.0 ** -149
    ref = np.array([1.0, 1.0, -3.0, 0.6 * sub, 0.6 * sub])
    got = np.array([1.0 + 0.9e-6, 1.0 + 1.1e-6, -3.0, sub, 2 * sub], np.float32)
    assert tol.accepted(got, F32, ref).tolist() == [True, False, True, True, False]
    assert tol.accepted(got[1:2], F32, ref[1:2], bound=2e-6).all()
    # relative to the terms' magnitude, not to a cancelled result
    assert tol.accepted(np.array([1e-7], np.float32), F32, np.array([0.0]), mag=0.2).all()
    b = oracle.store(np.array([1.0 + 7e-3, 1.0 + 1.2e-2]), BF16)  # 1 + 2^-7, 1 + 2^-6
    assert tol.accepted(b, BF16, np.array([1.0, 1.0])).tolist() == [True, False]


def _fp32_tree(a):
    a = list(np.asarray(a, np.float32))
    w = 1
    while w < len(a):
        for i in range(0, len(a) - w, 2 * w):
            a[i] = np.float32(a[i] + a[i + w])
        w *= 2
    return a[0]


def test_rmsnorm_bound_holds_for_a_simulated_fp32_row():
    hidden = 4096
    x = workloads.normal((1, hidden), 0, 1, 31, F32)[0]
    r = workloads.normal((1, hidden), 0, 1, 32, F32)[0]
    w = workloads.normal(hidden, 1, 0.1, 33, F32)
    y, _ = oracle.rmsnorm_residual(x[None], r[None], w, F32, 1e-6)
    h = (x + r).astype(np.float32)
    ss = _fp32_tree((h * h).astype(np.float32))
    rstd = np.float32(1) / np.sqrt(np.float32(ss / np.float32(hidden) + np.float32(1e-6)))
    dev = ((h * rstd).astype(np.float32) * w).astype(np.float32)
    rel = tol.rmsnorm_rel_bound(hidden)
    assert rel < 1e-6
    assert tol.accepted(dev, F32, y[0], bound=rel * np.abs(y[0])).all()
    # a device 5e-6 off in its row scale fails
    assert not tol.accepted((dev * np.float32(1 + 5e-6)).astype(np.float32), F32, y[0],
                            bound=rel * np.abs(y[0])).all()


def test_layernorm_bound_holds_for_a_simulated_fp32_row():
    hidden, eps = 1000, 1e-5
    x = workloads.normal((1, hidden), 0.5, 1, 41, F32)
    g = workloads.normal(hidden, 1, 0.2, 42, F32)
    b = workloads.normal(hidden, 0, 0.5, 43, F32)
    y, _, mag = oracle.layernorm_residual(x, None, g, b, F32, eps)
    h = x[0]
    mean = np.float32(_fp32_tree(h) / np.float32(hidden))
    d = (h - mean).astype(np.float32)
    var = np.float32(_fp32_tree((d * d).astype(np.float32)) / np.float32(hidden))
    rstd = np.float32(1) / np.sqrt(np.float32(var + np.float32(eps)))
    dev = ((d * rstd).astype(np.float32) * g + b).astype(np.float32)
    E = tol.layernorm_bound(oracle.to_double(x, F32), oracle.to_double(g, F32), y, eps)
    assert tol.accepted(dev, F32, y[0], mag[0], E[0]).all()
    # a mean off by 1e-4 fails
    bad = (((h - (mean + np.float32(1e-4))) * rstd).astype(np.float32) * g + b).astype(np.float32)
    assert not tol.accepted(bad, F32, y[0], mag[0], E[0]).all()


def test_reduction_depth_covers_the_kernels_trees():
    # ceil(log2 n) + 3: a row of 4096 in 256 threads of 16 is 4 + 5 + 3 = 12
    assert tol.reduction_depth(4096) == 15 and tol.reduction_depth(1) == 3
    assert tol.rmsnorm_rel_bound(1 << 15) < 1e-6 < tol.rmsnorm_rel_bound(1 << 16) < 1.02e-6
