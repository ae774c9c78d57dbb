"""GPU parity of the fixed entry points (rmsnorm_residual, layernorm_residual,
rope_qkv_split, detect_decode) against the fp64 oracle, through the C ABI.

Tolerances (tests/tolerance.py): bf16 outputs within 8e-3 relative, fp16
outputs within 2 ulp, fp32 outputs within 1e-6 relative -- relative to the
sum of the magnitudes of the terms where a result is a difference (a
rotation, h - mean, 2p - 0.5 + x) -- or within the derived worst-case bound
of the kernel's fp32 arithmetic where that is larger (long LayerNorm rows,
RMSNorm rows of 2^16).  Pure copies (v, the updated residual) are bit-exact.
Full-size workloads are checked on sampled rows/tokens.
"""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads
import tolerance as tol
from gpu_util import Guarded, misaligned_copy, to_dev, to_host

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------ RMSNorm

def _rms_case(rows, hidden, dt, seed, offset=0, inplace=False, eps=1e-6):
    x = workloads.normal((rows, hidden), 0, 1, seed, dt)
    r = workloads.normal((rows, hidden), 0, 1, seed + 1, dt)
    w = workloads.normal(hidden, 1, 0.1, seed + 2, dt)
    xd, rd, wd = (to_dev(a.reshape(-1), dt) for a in (x, r, w))
    if offset:
        xd, rd, wd = (misaligned_copy(t, offset) for t in (xd, rd, wd))
    out = Guarded(rows * hidden, dt, offset_elems=offset)
    if inplace:
        F.rmsnorm_residual(xd, rd, wd, out.t, rd, eps, dt, rows=rows, hidden=hidden)
        res_out_t = rd
    else:
        ro = Guarded(rows * hidden, dt, offset_elems=offset)
        F.rmsnorm_residual(xd, rd, wd, out.t, ro.t, eps, dt, rows=rows, hidden=hidden)
        res_out_t = ro.t
    torch.cuda.synchronize()
    assert out.canary_ok()
    y, h = oracle.rmsnorm_residual(x, r, w, dt, eps)
    got_r = to_host(res_out_t, dt).reshape(rows, hidden)
    assert np.array_equal(got_r, oracle.store(h, dt))  # one rounding of an exact sum
    tol.assert_accepted(to_host(out.t, dt), dt, y,
                        bound=tol.rmsnorm_rel_bound(hidden) * np.abs(y), what="rmsnorm y")


@pytest.mark.parametrize("rows,hidden", [(3, 4096), (67, 4096), (5, 1000), (4, 7), (2, 65536),
                                         (9, 8192), (1, 1)])
@pytest.mark.parametrize("dt", [F.BF16, F.F16, F.F32])
def test_rmsnorm_shapes(rows, hidden, dt):
    _rms_case(rows, hidden, dt, 100 + hidden % 97)


def test_rmsnorm_unaligned_and_in_place():
    _rms_case(11, 4096, F.BF16, 5, offset=1)
    _rms_case(11, 4096, F.BF16, 6, inplace=True)


def test_rmsnorm_unit_weight_rms_is_one():
    rows, hidden = 256, 4096
    x = workloads.normal((rows, hidden), 0, 1, 41, F.BF16)
    r = workloads.normal((rows, hidden), 0, 1, 42, F.BF16)
    w = oracle.store(np.ones(hidden), F.BF16)
    out = torch.empty(rows * hidden, dtype=torch.bfloat16, device="cuda")
    ro = torch.empty_like(out)
    F.rmsnorm_residual(to_dev(x.reshape(-1), F.BF16), to_dev(r.reshape(-1), F.BF16),
                       to_dev(w, F.BF16), out, ro, 1e-6, F.BF16, rows=rows, hidden=hidden)
    y = out.float().view(rows, hidden).double()
    rms = torch.sqrt((y * y).mean(dim=1))
    # bf16 rounding of each element moves the row RMS by well under 2^-9
    assert torch.all((rms - 1).abs() < 2e-3), rms


def test_rmsnorm_full_config_sampled_rows():
    cfg = workloads.RMSNORM
    rows, hidden = cfg["rows"], cfg["hidden"]
    x = workloads.device_normal((rows, hidden), 0, 1, cfg["seed"], F.BF16)
    r = workloads.device_normal((rows, hidden), 0, 1, cfg["seed"] + 1, F.BF16)
    w = workloads.device_normal((hidden,), 1, 0.1, cfg["seed"] + 2, F.BF16)
    out = torch.empty_like(x)
    ro = torch.empty_like(x)
    F.rmsnorm_residual(x, r, w, out, ro, cfg["eps"], F.BF16)
    torch.cuda.synchronize()
    g = np.random.default_rng(3)
    sel = np.unique(np.concatenate([[0, 1, rows - 1], g.integers(0, rows, 61)]))
    st = torch.from_numpy(sel).cuda()
    xs, rs = to_host(x[st], F.BF16), to_host(r[st], F.BF16)
    y, h = oracle.rmsnorm_residual(xs, rs, to_host(w, F.BF16), F.BF16, cfg["eps"])
    assert np.array_equal(to_host(ro[st], F.BF16), oracle.store(h, F.BF16))
    tol.assert_accepted(to_host(out[st], F.BF16), F.BF16, y, what="rmsnorm y")


# ------------------------------------------------------------ LayerNorm

def _ln_case(rows, hidden, dt, seed, flags=7, offset=0, inplace=False, eps=1e-5):
    has_res, has_g, has_b = bool(flags & 1), bool(flags & 2), bool(flags & 4)
    x = workloads.normal((rows, hidden), 0.5, 1, seed, dt)
    r = workloads.normal((rows, hidden), 0, 1, seed + 1, dt) if has_res else None
    g = workloads.normal(hidden, 1, 0.2, seed + 2, dt) if has_g else None
    b = workloads.normal(hidden, 0, 0.5, seed + 3, dt) if has_b else None
    dev = [None if a is None else to_dev(a.reshape(-1), dt) for a in (x, r, g, b)]
    if offset:
        dev = [None if t is None else misaligned_copy(t, offset) for t in dev]
    xd, rd, gd, bd = dev
    out = Guarded(rows * hidden, dt, offset_elems=offset)
    ro = None
    if has_res:
        ro = rd if inplace else Guarded(rows * hidden, dt, offset_elems=offset).t
    F.layernorm_residual(xd, rd, gd, bd, out.t, ro, eps, dt, rows=rows, hidden=hidden)
    torch.cuda.synchronize()
    assert out.canary_ok()
    y, h, mag = oracle.layernorm_residual(x, r, g, b, dt, eps)
    hx = oracle.to_double(x, dt) + (oracle.to_double(r, dt) if has_res else 0.0)
    if has_res:
        assert np.array_equal(to_host(ro, dt).reshape(rows, hidden), oracle.store(h, dt))
    E = tol.layernorm_bound(hx, None if g is None else oracle.to_double(g, dt), y, eps)
    tol.assert_accepted(to_host(out.t, dt), dt, y, mag, E, what="layernorm y")


@pytest.mark.parametrize("rows,hidden", [(3, 4096), (67, 4096), (5, 1000), (4, 7), (2, 65536),
                                         (1, 1), (9, 768)])
@pytest.mark.parametrize("dt", [F.BF16, F.F16, F.F32])
def test_layernorm_shapes(rows, hidden, dt):
    _ln_case(rows, hidden, dt, 300 + hidden % 89)


@pytest.mark.parametrize("flags", [0, 1, 2, 4, 3, 5, 6, 7])
def test_layernorm_optional_operands(flags):
    _ln_case(13, 2048, F.BF16, 40 + flags, flags=flags)


def test_layernorm_unaligned_and_in_place():
    _ln_case(11, 4096, F.BF16, 50, offset=1)
    _ln_case(11, 4096, F.BF16, 51, inplace=True)


def test_layernorm_full_config_sampled_rows():
    rows, hidden, eps = 16384, 4096, 1e-5
    x = workloads.device_normal((rows, hidden), 0, 1, 61, F.BF16)
    r = workloads.device_normal((rows, hidden), 0, 1, 62, F.BF16)
    g = workloads.device_normal((hidden,), 1, 0.1, 63, F.BF16)
    b = workloads.device_normal((hidden,), 0, 0.1, 64, F.BF16)
    out, ro = torch.empty_like(x), torch.empty_like(x)
    F.layernorm_residual(x, r, g, b, out, ro, eps, F.BF16)
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(5).integers(0, rows, 62)]))
    st = torch.from_numpy(sel).cuda()
    y, h, mag = oracle.layernorm_residual(to_host(x[st], F.BF16), to_host(r[st], F.BF16),
                                          to_host(g, F.BF16), to_host(b, F.BF16), F.BF16, eps)
    assert np.array_equal(to_host(ro[st], F.BF16), oracle.store(h, F.BF16))
    tol.assert_accepted(to_host(out[st], F.BF16), F.BF16, y, mag, what="layernorm y")


# ------------------------------------------------------------ many rows
# Thousands of rows: every SM runs many CTAs; tiny rows (24 elements) leave
# most lanes of a CTA idle; 480,000 f16 outputs reach below the smallest
# normal, where only the absolute tolerance holds.

MANY_ROWS = [(F.BF16, 4096, 3000), (F.F32, 1000, 6000), (F.F16, 24, 20000)]


@pytest.mark.parametrize("dt,hidden,rows", MANY_ROWS)
def test_rmsnorm_many_rows(dt, hidden, rows):
    _rms_case(rows, hidden, dt, 70)


@pytest.mark.parametrize("dt,hidden,rows", MANY_ROWS)
@pytest.mark.parametrize("flags", [7, 0])
def test_layernorm_many_rows(dt, hidden, rows, flags):
    _ln_case(rows, hidden, dt, 80, flags=flags)


def test_norms_in_place_many_rows():
    _rms_case(2000, 4096, F.BF16, 90, inplace=True)
    _ln_case(2000, 4096, F.BF16, 91, inplace=True)


# ------------------------------------------------------------ QKV split + RoPE

def _rope_check(qkv_host, heads, hd, pos0, dt, got_q, got_k, got_v, tokens_idx=None, base=1e4):
    tokens = qkv_host.shape[0]
    pos = pos0 + (np.arange(tokens) if tokens_idx is None else tokens_idx)
    q, k, v, qm, km = oracle.rope_qkv_split(qkv_host, dt, heads, hd, pos, base)
    for which, (got, want, mag) in enumerate(((got_q, q, qm), (got_k, k, km))):
        E = tol.rope_bound(mag, tol.rope_pair_abs(qkv_host, dt, heads, hd, which), pos)
        tol.assert_accepted(got, dt, want, mag, E, what="rope " + "qk"[which])
    assert np.array_equal(got_v.reshape(v.shape), oracle.store(v, dt))


@pytest.mark.parametrize("tokens,heads,hd,pos0", [
    (5, 4, 128, 0), (37, 3, 64, 32000), (8, 2, 80, 7), (3, 1, 6, 100), (16, 32, 128, 32752),
    (2, 2, 256, 1_000_000), (4, 3, 2, 5),  # head_dim 2: one rotation pair
])
@pytest.mark.parametrize("dt", [F.BF16, F.F16, F.F32])
def test_rope_shapes(tokens, heads, hd, pos0, dt):
    qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, tokens + hd, dt)
    qd = to_dev(qkv.reshape(-1), dt)
    outs = [Guarded(heads * tokens * hd, dt) for _ in range(3)]
    F.rope_qkv_split(qd, outs[0].t, outs[1].t, outs[2].t, heads, hd, pos0, 10000.0, dt,
                     tokens=tokens)
    torch.cuda.synchronize()
    assert all(o.canary_ok() for o in outs)
    _rope_check(qkv, heads, hd, pos0, dt, *(to_host(o.t, dt) for o in outs))


@pytest.mark.parametrize("tokens,heads,hd,pos0,dt", [
    (4, 96, 128, 0, F.F16),        # 3 q/k items a thread: 3 rounds
    (3, 160, 256, 5, F.F32),       # 20 rounds
    (2, 1024, 1024, 11, F.BF16),   # the widest row the entry point takes: heads * head_dim = 2^20
])
def test_rope_wide_rows(tokens, heads, hd, pos0, dt):
    """Rows with more q/k items than one round of a thread's registers holds
    run in several rounds of the same kernel."""
    qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, 3 * tokens + heads, dt)
    qd = to_dev(qkv.reshape(-1), dt)
    outs = [Guarded(heads * tokens * hd, dt) for _ in range(3)]
    F.rope_qkv_split(qd, outs[0].t, outs[1].t, outs[2].t, heads, hd, pos0, 10000.0, dt,
                     tokens=tokens)
    torch.cuda.synchronize()
    assert all(o.canary_ok() for o in outs)
    _rope_check(qkv, heads, hd, pos0, dt, *(to_host(o.t, dt) for o in outs))


def test_rope_unaligned_and_position_zero_identity():
    tokens, heads, hd, dt = 9, 4, 128, F.BF16
    qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, 77, dt)
    qd = misaligned_copy(to_dev(qkv.reshape(-1), dt), 1)
    outs = [Guarded(heads * tokens * hd, dt, offset_elems=1) for _ in range(3)]
    F.rope_qkv_split(qd, outs[0].t, outs[1].t, outs[2].t, heads, hd, 0, 10000.0, dt, tokens=tokens)
    torch.cuda.synchronize()
    assert all(o.canary_ok() for o in outs)
    got = [to_host(o.t, dt) for o in outs]
    _rope_check(qkv, heads, hd, 0, dt, *got)
    # token 0 is at position 0: q and k are copied exactly
    src = qkv.reshape(tokens, 3, heads, hd)
    assert np.array_equal(got[0].reshape(heads, tokens, hd)[:, 0], src[0, 0])
    assert np.array_equal(got[1].reshape(heads, tokens, hd)[:, 0], src[0, 1])


def test_rope_full_config_sampled_tokens():
    cfg = workloads.ROPE
    T, H, D = cfg["tokens"], cfg["heads"], cfg["head_dim"]
    qkv = workloads.device_normal((T, 3 * H * D), 0, 1, cfg["seed"], F.BF16)
    q = torch.empty(H * T * D, dtype=torch.bfloat16, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    F.rope_qkv_split(qkv, q, k, v, H, D, cfg["pos0"], cfg["base"], F.BF16)
    torch.cuda.synchronize()
    g = np.random.default_rng(4)
    sel = np.unique(np.concatenate([[0, 1, T - 1], g.integers(0, T, 61)]))
    st = torch.from_numpy(sel).cuda()
    sub = lambda t: to_host(t.view(H, T, D)[:, st].contiguous(), F.BF16)  # noqa: E731
    _rope_check(to_host(qkv[st], F.BF16), H, D, cfg["pos0"], F.BF16, sub(q), sub(k), sub(v),
                tokens_idx=sel)


def _table_check(fn, tokens, pos0, hd=128):
    """The cos/sin values a RoPE entry point uses, read back exactly: fp32 q
    rows of ones then zeros rotate to (cos theta_i, sin theta_i) and k rows of
    zeros then ones to (-sin theta_i, cos theta_i), with no rounding in the
    rotation (products by 1 and 0).  Each must be within one ulp of the fp32
    value nearest the oracle's cos or sin, or within the error of the angle
    itself: both sides form theta = pos * base^(-2i/D) in binary64, which is
    good to about pos * 2^-52 radians, and near a zero of cos or sin that
    absolute error is many fp32 ulps (bound used: pos * 2^-50).  Where that
    error is near an fp32 rounding step the two sides round apart, about one
    value in 10^3 at positions near 2^22; at most 1 % may."""
    half = hd // 2
    qkv = np.zeros((tokens, 3, 1, hd), np.float32)
    qkv[:, 0, 0, :half] = 1.0
    qkv[:, 1, 0, half:] = 1.0
    outs = [torch.empty(tokens * hd, dtype=torch.float32, device="cuda") for _ in range(3)]
    fn(to_dev(qkv.reshape(-1), F.F32), *outs, 1, hd, pos0, 10000.0, F.F32, tokens=tokens)
    torch.cuda.synchronize()
    q, k, _, _, _ = oracle.rope_qkv_split(qkv.reshape(tokens, -1), F.F32, 1, hd,
                                         pos0 + np.arange(tokens))
    def order(a):  # monotone integer image of fp32 values (both zeros map to 0)
        b = a.view(np.int32).astype(np.int64)
        return np.where(b < 0, -(b & 0x7FFFFFFF), b)
    theta_err = np.repeat((pos0 + np.arange(tokens)) * 2.0 ** -50, hd)
    for got, want in ((outs[0], q), (outs[1], k)):
        g = to_host(got, F.F32)
        w = want.reshape(-1)
        d = np.abs(order(g) - order(oracle.store(w, F.F32)))
        ok = (d <= 1) | (np.abs(g.astype(np.float64) - w) <= theta_err)
        assert ok.all() and (d > 0).mean() <= 1e-2, (int((~ok).sum()), int((d > 0).sum()))


@pytest.mark.parametrize("pos0", [0, 1000, (1 << 22) - 2048])
def test_rope_table_is_correctly_rounded(pos0):
    _table_check(F.rope_qkv_split, 2048, pos0)


# ------------------------------------------------------------ detection decode

def _detect_case(hw, dt, seed, offset=0, na=3, no=85):
    strides = [8.0 * 2 ** s for s in range(len(hw))]
    anchors = workloads.detect_anchors(strides, na)
    feats = [workloads.normal((1, na * no, h, w), 0, 2.0, seed + s, dt) for s, (h, w) in enumerate(hw)]
    fd = [to_dev(f.reshape(-1), dt) for f in feats]
    if offset:
        fd = [misaligned_copy(t, offset) for t in fd]
    rows = sum(na * h * w for h, w in hw)
    out = Guarded(rows * no, F.F32, offset_elems=offset)
    F.detect_decode(fd, hw, strides, anchors, na, no, out.t, dt)
    torch.cuda.synchronize()
    assert out.canary_ok()
    want, mag = oracle.detect_decode(feats, dt, strides, anchors, na, no)
    tol.assert_accepted(to_host(out.t, F.F32), F.F32, want, mag, what="detect")


def test_detect_full_config():
    cfg = workloads.DETECT
    _detect_case(cfg["hw"], F.F16, cfg["seed"])


def test_detect_decoder_object_matches_the_function():
    """DetectDecoder converts the fixed arguments once; its calls give the
    same bits as detect_decode on the same inputs, frame after frame."""
    cfg = workloads.DETECT
    hw, na, no = cfg["hw"], cfg["na"], cfg["no"]
    anchors = workloads.detect_anchors(cfg["strides"], na)
    rows = sum(na * h * w for h, w in hw)
    dec = F.DetectDecoder(hw, cfg["strides"], anchors, na, no, F.F16)
    for frame in range(3):
        feats = [workloads.device_normal((1, na * no, h, w), 0, 2.0, 70 + 3 * frame + s, F.F16,
                                         "cuda") for s, (h, w) in enumerate(hw)]
        a = torch.empty(rows * no, dtype=torch.float32, device="cuda")
        b = torch.empty_like(a)
        dec(feats, a)
        F.detect_decode(feats, hw, cfg["strides"], anchors, na, no, b, F.F16)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


@pytest.mark.parametrize("hw", [[(1, 1)], [(3, 3), (2, 1), (1, 2)], [(8, 8), (4, 4), (2, 2)],
                                [(13, 7), (5, 9)], [(80, 80), (40, 40), (20, 20), (10, 10)]])
@pytest.mark.parametrize("dt", [F.F16, F.F32, F.BF16])
def test_detect_shapes(hw, dt):
    _detect_case(hw, dt, 11)


@pytest.mark.parametrize("hw,dt,na,no", [
    ([(16, 16), (8, 8), (4, 4)], F.F16, 3, 85),  # 32-byte vectors: 16 cells a warp
    ([(8, 8), (4, 2)], F.F16, 3, 85),            # a plane of 8 cells: 16-byte vectors
    ([(16, 16), (8, 8)], F.F32, 3, 85),
    ([(24, 8)], F.BF16, 2, 6),
    ([(16, 16)], F.F16, 1, 128),                 # four channels a lane
    ([(4, 4), (2, 2)], F.F32, 4, 37),
])
def test_detect_other_heads_and_vector_planes(hw, dt, na, no):
    """Planes of whole 16- and 32-byte input vectors, fp32 and bf16 inputs, and
    heads of 6 to 128 outputs with one to four anchors."""
    _detect_case(hw, dt, 21, na=na, no=no)


def test_detect_unaligned_and_other_heads():
    _detect_case([(16, 16), (8, 8)], F.F16, 12, offset=1)
    _detect_case([(10, 12)], F.F16, 13, na=2, no=6)
    _detect_case([(4, 6)], F.F32, 14, na=1, no=1024)


def test_detect_sigmoid_zero_closed_form():
    hw = [(8, 8), (4, 4), (2, 2)]
    strides = [8.0, 16.0, 32.0]
    anchors = workloads.detect_anchors(strides)
    fd = [torch.zeros(255 * h * w, dtype=torch.float16, device="cuda") for h, w in hw]
    rows = sum(3 * h * w for h, w in hw)
    out = torch.empty(rows * 85, dtype=torch.float32, device="cuda")
    F.detect_decode(fd, hw, strides, anchors, 3, 85, out, F.F16)
    o = out.view(rows, 85).cpu().numpy()
    assert np.all(o[:, 4:] == 0.5)
    assert o[0, 0] == 4.0 and o[0, 1] == 4.0 and o[0, 2] == anchors[0, 0, 0]
    assert o[3 * 64, 0] == 8.0  # first row of scale 1: (0.5 + 0) * 16


# ------------------------------------------------------------ zero-size calls

def test_zero_size_calls_launch_nothing_and_write_nothing():
    """rows = 0, tokens = 0 and a batch of 0 are valid calls: they return
    without a launch and leave every output byte as it was."""
    dt = F.BF16
    buf = [torch.full((4096,), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    before = [b.clone() for b in buf]
    stats = F.fuse_stats()
    F.rmsnorm_residual(buf[0], buf[1], buf[2], buf[3], buf[4], 1e-6, dt, rows=0, hidden=4096)
    F.layernorm_residual(buf[0], buf[1], buf[2], buf[5], buf[3], buf[4], 1e-5, dt, rows=0,
                         hidden=4096)
    F.rope_qkv_split(buf[0], buf[3], buf[4], buf[5], 4, 128, 0, 10000.0, dt, tokens=0)
    F.rope_qkv_split_noalloc(buf[0], buf[3], buf[4], buf[5], 4, 128, 0, 10000.0, dt, tokens=0)
    F.channel_shuffle(buf[0], buf[3], 4, dt, shape=(0, 16, 8, 8))
    torch.cuda.synchronize()
    assert F.fuse_stats()["launches"] == stats["launches"]
    assert all(torch.equal(a, b) for a, b in zip(buf, before))
