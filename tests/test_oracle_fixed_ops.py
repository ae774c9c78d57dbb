"""Pins for the oracle's ChannelShuffle, residual-add + RMSNorm, QKV split +
RoPE and detection-head decode (CPU only).

Each pin is something the pages or the mathematics fix independently of the
oracle's code: index brute force against numpy reshape/transpose, round trips,
closed forms (constant rows, one-hot rotations, sigmoid(0) = 1/2), and
invariants (unit-weight RMS, rotation norms, relative-position dot products).
"""
import math

import numpy as np
import pytest

import oracle
import workloads


# ------------------------------------------------------------ ChannelShuffle
# "算子与运行时" section 2: reshape(n, g, c/g, h, w) -> transpose(1, 2) -> reshape

@pytest.mark.parametrize("shape", [(2, 8, 3, 3), (1, 12, 1, 5), (3, 6, 2, 1)])
def test_shuffle_index_brute_force(shape):
    n, c, h, w = shape
    x = np.arange(np.prod(shape), dtype=np.int32).reshape(shape)  # value = flat index
    for g in [d for d in range(1, c + 1) if c % d == 0]:
        got = oracle.channel_shuffle(x, g)
        want = x.reshape(n, g, c // g, h, w).transpose(0, 2, 1, 3, 4).reshape(shape)
        assert np.array_equal(got, want), g


def test_shuffle_round_trip_with_inverse_groups():
    x = workloads.uniform((4, 24, 5, 7), -2, 2, 21, oracle.F16)
    for g in (2, 3, 4, 6, 8, 12):
        y = oracle.channel_shuffle(x, g)
        assert not np.array_equal(y, x)
        assert np.array_equal(oracle.channel_shuffle(y, 24 // g), x)


def test_shuffle_trivial_groups_are_identity():
    x = workloads.uniform((2, 16, 3, 3), -2, 2, 22, oracle.F16)
    assert np.array_equal(oracle.channel_shuffle(x, 1), x)
    assert np.array_equal(oracle.channel_shuffle(x, 16), x)


def test_shuffle_moves_whole_planes():
    x = workloads.uniform((2, 8, 4, 4), -2, 2, 23, oracle.F32)
    y = oracle.channel_shuffle(x, 4)
    for co in range(8):
        ci = (co % 4) * 2 + co // 4
        assert np.array_equal(y[:, co], x[:, ci])


# ------------------------------------------------------------ RMSNorm
# "TeleTron" sections 3.3 and 4.2: h = x + residual, rms scale
# rsqrt(sum(h^2)/K + eps), fp32-or-better accumulation.

def _bf16(values):
    return oracle.store(np.asarray(values, np.float64), oracle.BF16)


def test_rmsnorm_unit_weight_rows_have_unit_rms():
    rows, hidden, eps = 64, 4096, 1e-6
    x = workloads.normal((rows, hidden), 0, 1, 31, oracle.BF16)
    r = workloads.normal((rows, hidden), 0, 1, 32, oracle.BF16)
    w = _bf16(np.ones(hidden))
    y, h = oracle.rmsnorm_residual(x, r, w, oracle.BF16, eps)
    ms = np.mean(h * h, axis=1)
    rms_y = np.sqrt(np.mean(y * y, axis=1))
    # exact identity: rms(y) = sqrt(ms / (ms + eps)); within 1e-6 of 1 here
    np.testing.assert_allclose(rms_y, np.sqrt(ms / (ms + np.float32(eps))), rtol=1e-13)
    assert np.all(np.abs(rms_y - 1) < 1e-6)


def test_rmsnorm_constant_rows_closed_form():
    hidden, eps = 256, 1e-6
    cs = np.array([1.0, -2.0, 0.001, 3.5, -0.25])
    x = _bf16(np.repeat(cs[:, None], hidden, 1))
    r = _bf16(np.zeros((len(cs), hidden)))
    w = _bf16(np.linspace(0.5, 1.5, hidden))
    y, h = oracle.rmsnorm_residual(x, r, w, oracle.BF16, eps)
    cb = oracle.to_double(x[:, 0], oracle.BF16)
    wd = oracle.to_double(w, oracle.BF16)
    e32 = float(np.float32(eps))
    want = (cb / np.sqrt(cb * cb + e32))[:, None] * wd[None, :]
    np.testing.assert_allclose(y, want, rtol=1e-14)
    # c = 0.001 (in bf16) makes eps matter: y = c / sqrt(c^2 + eps) is near 0.7
    assert abs(y[2, 0] / wd[0] - cb[2] / math.sqrt(cb[2] ** 2 + e32)) < 1e-14
    assert 0.6 < y[2, 0] / wd[0] < 0.8


def test_rmsnorm_zero_row_gives_zero():
    x = _bf16(np.zeros((2, 128)))
    w = _bf16(np.ones(128))
    y, h = oracle.rmsnorm_residual(x, x, w, oracle.BF16, 1e-6)
    assert np.all(y == 0) and np.all(h == 0)


def test_rmsnorm_residual_out_is_the_exact_sum():
    g = np.random.default_rng(33)
    a = g.integers(-100, 100, (8, 64)).astype(np.float64)
    b = g.integers(-100, 100, (8, 64)).astype(np.float64)
    y, h = oracle.rmsnorm_residual(_bf16(a), _bf16(b), _bf16(np.ones(64)), oracle.BF16, 1e-6)
    assert np.array_equal(h, a + b)  # integers < 256 in magnitude are exact in bf16


def test_rmsnorm_scale_invariance_and_weight_linearity():
    x = workloads.normal((16, 512), 0, 1, 34, oracle.BF16)
    r = workloads.normal((16, 512), 0, 1, 35, oracle.BF16)
    w = workloads.normal(512, 1, 0.1, 36, oracle.BF16)
    y, _ = oracle.rmsnorm_residual(x, r, w, oracle.BF16, 0.0)
    xd, rd = oracle.to_double(x, oracle.BF16), oracle.to_double(r, oracle.BF16)
    y4, _ = oracle.rmsnorm_residual(_bf16(4 * xd), _bf16(4 * rd), w, oracle.BF16, 0.0)
    np.testing.assert_allclose(y4, y, rtol=1e-14)  # power-of-two scaling is exact in bf16
    wd = oracle.to_double(w, oracle.BF16)
    y2, _ = oracle.rmsnorm_residual(x, r, _bf16(2 * wd), oracle.BF16, 0.0)
    np.testing.assert_allclose(y2, 2 * y, rtol=1e-15)


def test_rmsnorm_rows_are_independent_and_permutation_equivariant():
    x = workloads.normal((4, 300), 0, 1, 37, oracle.BF16)
    r = workloads.normal((4, 300), 0, 1, 38, oracle.BF16)
    w = _bf16(np.ones(300))
    y, _ = oracle.rmsnorm_residual(x, r, w, oracle.BF16, 1e-6)
    perm = np.random.default_rng(39).permutation(300)
    yp, _ = oracle.rmsnorm_residual(x[:, perm], r[:, perm], w, oracle.BF16, 1e-6)
    np.testing.assert_allclose(yp, y[:, perm], rtol=1e-14)
    y1, _ = oracle.rmsnorm_residual(x[2:3], r[2:3], w, oracle.BF16, 1e-6)
    assert np.array_equal(y1[0], y[2])


# ------------------------------------------------------------ QKV split + RoPE
# rotate-half RoPE, base 10000, on q and k; v copied; [T,3,H,D] -> [H,T,D]

H, D = 4, 128


def _qkv(tokens, seed):
    return workloads.normal((tokens, 3 * H * D), 0, 1, seed, oracle.BF16)


def test_rope_position_zero_is_identity_and_split_indexing():
    T = 5
    vals = np.arange(T * 3 * H * D) % 251 - 125  # small integers: exact in bf16
    qkv = _bf16(vals.reshape(T, 3 * H * D))
    q, k, v, _, _ = oracle.rope_qkv_split(qkv, oracle.BF16, H, D, np.zeros(T, np.int64))
    src = vals.reshape(T, 3, H, D).astype(np.float64)
    assert np.array_equal(q, src[:, 0].transpose(1, 0, 2))
    assert np.array_equal(k, src[:, 1].transpose(1, 0, 2))
    assert np.array_equal(v, src[:, 2].transpose(1, 0, 2))


def test_rope_one_hot_rotation_closed_form():
    pos = np.array([0, 1, 7, 100, 32767], np.int64)
    for i in (0, 32, 63):
        qkv = np.zeros((len(pos), 3, H, D))
        qkv[:, 0, :, i] = 1.0            # q = e_i
        qkv[:, 1, :, i + D // 2] = 1.0   # k = e_{i+64}
        q, k, _, _, _ = oracle.rope_qkv_split(_bf16(qkv.reshape(len(pos), -1)), oracle.BF16,
                                              H, D, pos)
        inv_freq = {0: 1.0, 32: 0.01, 63: 10000.0 ** (-126 / 128)}[i]
        th = pos * inv_freq
        # e_i -> cos at i, +sin at i + 64;  e_{i+64} -> -sin at i, cos at i + 64
        np.testing.assert_allclose(q[:, :, i], np.broadcast_to(np.cos(th), (H, len(pos))), atol=1e-12)
        np.testing.assert_allclose(q[:, :, i + 64], np.broadcast_to(np.sin(th), (H, len(pos))), atol=1e-12)
        np.testing.assert_allclose(k[:, :, i], np.broadcast_to(-np.sin(th), (H, len(pos))), atol=1e-12)
        np.testing.assert_allclose(k[:, :, i + 64], np.broadcast_to(np.cos(th), (H, len(pos))), atol=1e-12)


def test_rope_preserves_pair_norms():
    T = 16
    qkv = _qkv(T, 41)
    pos = np.arange(T, dtype=np.int64) * 2047
    q, k, _, _, _ = oracle.rope_qkv_split(qkv, oracle.BF16, H, D, pos)
    src = oracle.to_double(qkv, oracle.BF16).reshape(T, 3, H, D)
    for out, which in ((q, 0), (k, 1)):
        x = src[:, which].transpose(1, 0, 2)
        n_in = np.hypot(x[..., :64], x[..., 64:])
        n_out = np.hypot(out[..., :64], out[..., 64:])
        np.testing.assert_allclose(n_out, n_in, rtol=1e-13, atol=1e-13)


def test_rope_relative_position_property():
    qkv = _qkv(1, 42)
    dots = []
    for m, n in ((5, 2), (103, 100), (32000, 31997)):
        qm, _, _, _, _ = oracle.rope_qkv_split(qkv, oracle.BF16, H, D, np.array([m]))
        _, kn, _, _, _ = oracle.rope_qkv_split(qkv, oracle.BF16, H, D, np.array([n]))
        dots.append(np.sum(qm[:, 0] * kn[:, 0], axis=-1))
    np.testing.assert_allclose(dots[1], dots[0], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(dots[2], dots[0], rtol=1e-9, atol=1e-9)


def test_rope_v_is_bit_copy():
    qkv = _qkv(7, 43)
    _, _, v, _, _ = oracle.rope_qkv_split(qkv, oracle.BF16, H, D, np.arange(7) + 1000)
    src = qkv.reshape(7, 3, H, D)[:, 2].transpose(1, 0, 2)
    assert np.array_equal(oracle.store(v, oracle.BF16), src)


# ------------------------------------------------------------ detection decode

def _anchors():
    return workloads.detect_anchors([8.0, 16.0, 32.0])


def test_detect_sigmoid_zero_closed_form():
    hw = [(3, 2), (2, 2), (1, 1)]
    feats = [np.zeros((1, 255, h, w), np.uint16) for h, w in hw]  # fp16 +0
    out, _ = oracle.detect_decode(feats, oracle.F16, [8.0, 16.0, 32.0], _anchors(), 3, 85)
    anc = _anchors()
    row = 0
    for s, (h, w) in enumerate(hw):
        st = [8.0, 16.0, 32.0][s]
        for a in range(3):
            for y in range(h):
                for x in range(w):
                    assert out[row, 0] == (0.5 + x) * st
                    assert out[row, 1] == (0.5 + y) * st
                    assert out[row, 2] == anc[s, a, 0] and out[row, 3] == anc[s, a, 1]
                    assert np.all(out[row, 4:] == 0.5)
                    row += 1
    assert row == out.shape[0]


def test_detect_logit_recovers_source_index():
    # distinct logits per source element: logit(out[row, k]) for k >= 4 names
    # the (scale, channel, y, x) it came from
    hw = [(3, 3), (2, 1), (1, 1)]
    feats, code = [], {}
    nxt = 0
    for s, (h, w) in enumerate(hw):
        vals = np.zeros((1, 255, h, w))
        for c in range(255):
            for y in range(h):
                for x in range(w):
                    v = (nxt - 1530) * 2.0 ** -8  # distinct, exact in fp16 (|v| < 6)
                    vals[0, c, y, x] = v
                    code[v] = (s, c, y, x)
                    nxt += 1
        feats.append(oracle.store(vals, oracle.F16))
    out, _ = oracle.detect_decode(feats, oracle.F16, [8.0, 16.0, 32.0], _anchors(), 3, 85)
    offs = [0, 3 * 9, 3 * 9 + 3 * 2]
    assert out.shape[0] == 3 * 9 + 3 * 2 + 3 * 1
    for s, (h, w) in enumerate(hw):
        for a in range(3):
            for y in range(h):
                for x in range(w):
                    row = offs[s] + a * h * w + y * w + x
                    for k in (4, 40, 84):
                        p = out[row, k]
                        logit = math.log(p / (1 - p))
                        key = min(code, key=lambda v: abs(v - logit))
                        assert abs(key - logit) < 1e-9
                        assert code[key] == (s, a * 85 + k, y, x)


def test_detect_box_outputs_follow_the_class_outputs():
    # every channel of a cell carries the same logit, so the cell's box
    # outputs and its class outputs share one p, which the class outputs give
    # (pinned on their own above); then x / stride - grid_x + 0.5 = 2p,
    # likewise for y, and w / anchor_w = h / anchor_h = (2p)^2 -- away from
    # p = 1/2, where the zero-logit closed form cannot tell (2p)^2 from 2p
    hw = [(2, 3), (1, 2), (1, 1)]
    strides = [8.0, 16.0, 32.0]
    logits = [-3.0, -1.0, 0.5, 2.0, 1.25, -0.75]
    feats = []
    for s, (h, w) in enumerate(hw):
        vals = np.zeros((1, 255, h, w))
        for y in range(h):
            for x in range(w):
                vals[0, :, y, x] = logits[(s + y * w + x) % len(logits)]
        feats.append(oracle.store(vals, oracle.F16))
    anc = _anchors()
    out, _ = oracle.detect_decode(feats, oracle.F16, strides, anc, 3, 85)
    row = 0
    for s, (h, w) in enumerate(hw):
        for a in range(3):
            for y in range(h):
                for x in range(w):
                    p = out[row, 4]
                    assert np.all(out[row, 4:] == p) and 0.0 < p < 1.0 and p != 0.5
                    two_p = 2.0 * p
                    assert out[row, 0] / strides[s] - x + 0.5 == pytest.approx(two_p, rel=1e-12)
                    assert out[row, 1] / strides[s] - y + 0.5 == pytest.approx(two_p, rel=1e-12)
                    assert out[row, 2] / anc[s, a, 0] == pytest.approx(two_p ** 2, rel=1e-12)
                    assert out[row, 3] / anc[s, a, 1] == pytest.approx(two_p ** 2, rel=1e-12)
                    row += 1


def test_detect_concat_offsets_full_shapes():
    hw = [(80, 80), (40, 40), (20, 20)]
    rows = [3 * h * w for h, w in hw]
    assert np.cumsum([0] + rows)[:3].tolist() == [0, 19200, 24000]
    assert sum(rows) == 25200
