"""GPU parity of fused elementwise chains and ChannelShuffle against the oracle.

Every case runs through the C ABI (fuse_compile / fuse_launch /
channel_shuffle) on seeded inputs from `workloads`, and is compared element by
element with the fp64 oracle: bit-exact for add -> relu -> scale (whose exact
result is one fp32 rounding) and for the shuffle copies; the flat tolerance or
the oracle's running error bound for random chains.  Sizes span several
chunks plus ragged remainders and tails; odd offsets take the scalar kernel;
canary bytes after each output catch writes past the end.
"""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads
from gpu_util import Guarded, misaligned_copy, to_dev, to_host

pytestmark = pytest.mark.gpu


def _run_chain(spec, dt, inputs, shape, offset=0):
    c = F.fuse_compile(spec, shape, dt)
    dev = [to_dev(a, d) for a, d in zip(inputs, c.in_dtypes)]
    if offset:
        dev = [misaligned_copy(t, offset) for t in dev]
    n = int(np.prod(shape))
    out = Guarded(n, c.out_dtype, offset_elems=offset)
    F.fuse_launch(c, dev, out.t)
    torch.cuda.synchronize()
    assert out.canary_ok(), "write outside the output"
    return to_host(out.t, c.out_dtype), c


# ------------------------------------------------------------ add -> relu -> scale

@pytest.mark.parametrize("n", [1 << 20, 1, 7, 67, 4099, (1 << 20) + 7])
@pytest.mark.parametrize("offset", [0, 1])
def test_add_relu_scale_bit_exact(n, offset):
    cfg = workloads.ADD_RELU_SCALE
    a = workloads.uniform(n, cfg["lo"], cfg["hi"], cfg["seed"], F.F32)
    b = workloads.uniform(n, cfg["lo"], cfg["hi"], cfg["seed"] + 100, F.F32)
    got, _ = _run_chain(cfg["spec"], F.F32, [a, b], (n,), offset)
    want, _ = oracle.chain_eval(cfg["spec"], F.F32, [a, b], (n,))
    assert np.array_equal(got, oracle.store(want, F.F32))


def test_bound_launch_runs_the_chain_on_its_tensors():
    """Chain.bind: the same chain on the same tensors step after step, with
    new input values each step, bit-exact against the oracle's closed form."""
    cfg = workloads.ADD_RELU_SCALE
    n = (1 << 20) + 7
    c = F.fuse_compile(cfg["spec"], (n,), F.F32)
    a_t = torch.empty(n, dtype=torch.float32, device="cuda")
    b_t = torch.empty_like(a_t)
    out = Guarded(n, F.F32)
    step = c.bind([a_t, b_t], out.t)
    for k in range(3):
        a = workloads.uniform(n, cfg["lo"], cfg["hi"], 50 + k, F.F32)
        b = workloads.uniform(n, cfg["lo"], cfg["hi"], 60 + k, F.F32)
        a_t.copy_(torch.from_numpy(a))
        b_t.copy_(torch.from_numpy(b))
        step()
        torch.cuda.synchronize()
        assert out.canary_ok()
        want, _ = oracle.chain_eval(cfg["spec"], F.F32, [a, b], (n,))
        assert np.array_equal(to_host(out.t, F.F32), oracle.store(want, F.F32))


def test_longest_and_widest_chain():
    """The engine's limits at once: 1024 ops and 128 input tensors (127 adds),
    over the vector body, the remainder and the scalar tail, against the
    oracle.  Every exp follows a sigmoid, so the values stay bounded and the
    running error bound decides every element."""
    group = ["add", "sigmoid", "relu", "scale:0.75", "exp", "sigmoid", "scale:1.5", "relu"]
    tail = ["sigmoid", "exp", "relu", "scale:0.5", "sigmoid", "exp", "scale:0.25", "relu"]
    ops = group * 127 + tail
    spec = ";".join(ops)
    n = 4099
    inputs, _ = workloads.chain_inputs(spec, F.F32, n, 77)
    got, c = _run_chain(spec, F.F32, inputs, (n,))
    assert len(ops) == 1024 and c.n_in == 128
    _check(spec, F.F32, inputs, (n,), got)


def test_add_relu_scale_golden_on_device():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "add_relu_scale.txt")
    rows = [l.split("#", 1)[0].split() for l in open(path)]
    rows = [r for r in rows if r]
    num = lambda s: float.fromhex(s) if "0x" in s else float(s)  # noqa: E731
    a = np.array([num(r[0]) for r in rows], np.float32)
    b = np.array([num(r[1]) for r in rows], np.float32)
    want = np.array([num(r[2]) for r in rows], np.float32)
    got, _ = _run_chain("add;relu;scale:0.5", F.F32, [a, b], (len(a),))
    assert np.array_equal(got, want) and not np.any(np.signbit(got))


# ------------------------------------------------------------ every fp16 input, one op

@pytest.mark.parametrize("op", ["relu", "sigmoid", "exp", "scale:0.7529296875", "cast:bf16",
                                "exp:fast", "sigmoid:fast"])
@pytest.mark.parametrize("out", ["f16", "f32"])
def test_unary_op_on_every_fp16_value(op, out):
    """All 65,536 fp16 bit patterns (incl. subnormals, inf, NaN) through one
    op, stored as fp16 or (after a cast to fp32) as fp32."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    spec = op if out == "f16" else "cast:f32;" + op
    if op == "cast:bf16":
        spec = "cast:bf16" if out == "f16" else "cast:bf16;cast:f32"
    got, c = _run_chain(spec, F.F16, [x], x.shape)
    fails, counts, cls = oracle.chain_check(spec, F.F16, [x], x.shape, got)
    assert fails == 0, (spec, counts, x[cls == 2][:8])
    assert counts[3] == 0, (spec, counts)


@pytest.mark.parametrize("op", ["sigmoid", "exp", "sigmoid;sigmoid", "exp:fast", "sigmoid:fast",
                                "sigmoid:fast;sigmoid:fast", "exp:fast;scale:0.5;exp:fast"])
def test_transcendentals_over_the_fp32_range(op):
    """4M fp32 values spread over [-104, 104] plus the special values: where
    exp(-x) overflows, where 1 + exp(-x) passes 2^126 and the reciprocal
    flushes to zero, where exp underflows and overflows.  Every element is
    pinned (flat 1e-6 or the running bound), none unpinned."""
    grid = np.linspace(-104.0, 104.0, 1 << 22, dtype=np.float64).astype(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.4028235e38, -3.4028235e38, 1e-45,
                        -1e-45, 1.1754944e-38, -87.33655, -87.33654, 88.72283, 88.72284,
                        -103.97208, -103.97209], dtype=np.float32)
    x = np.concatenate([grid, special])
    got, _ = _run_chain(op, F.F32, [x], x.shape)
    fails, counts, cls = oracle.chain_check(op, F.F32, [x], x.shape, got)
    assert fails == 0, (op, counts, x[cls == 2][:8], got[cls == 2][:8])
    assert counts[3] == 0, (op, counts)


# ------------------------------------------------------------ random chains

def _check(spec, dt, inputs, shape, got, idx=None):
    fails, counts, cls = oracle.chain_check(spec, dt, inputs, shape, got, idx)
    assert fails == 0, (spec, counts, np.nonzero(cls == 2)[0][:10])
    # unpinned: elements whose error interval spans more outcomes than the
    # check follows; none are allowed
    assert counts[3] == 0, (spec, counts)
    return counts


@pytest.mark.parametrize("length", workloads.CHAIN_LENGTHS)
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("n", [1, 33, 4099, (1 << 16) + 7])
def test_random_chain_small(length, seed, n):
    spec, dt = workloads.random_chain(length, seed)
    inputs, _ = workloads.chain_inputs(spec, dt, n, seed)
    got, _ = _run_chain(spec, dt, inputs, (n,))
    _check(spec, dt, inputs, (n,), got)


@pytest.mark.parametrize("length", workloads.CHAIN_LENGTHS)
@pytest.mark.parametrize("seed", [0, 1])
def test_random_chain_with_fast_transcendentals(length, seed):
    """Random chains with every exp and sigmoid in its opt-in fast form, at
    2^16 + 7 elements, against the oracle's bound for the fast forms."""
    spec, dt = workloads.random_chain(length, seed)
    spec = ";".join("exp:fast" if o == "exp" else "sigmoid:fast" if o == "sigmoid" else o
                    for o in spec.split(";"))
    n = (1 << 16) + 7
    inputs, _ = workloads.chain_inputs(spec, dt, n, seed)
    got, _ = _run_chain(spec, dt, inputs, (n,))
    _check(spec, dt, inputs, (n,), got)


@pytest.mark.parametrize("length", [2, 8, 32])
def test_random_chain_unaligned(length):
    spec, dt = workloads.random_chain(length, 7)
    n = 10_007
    inputs, _ = workloads.chain_inputs(spec, dt, n, 7)
    got, _ = _run_chain(spec, dt, inputs, (n,), offset=1)
    _check(spec, dt, inputs, (n,), got)


@pytest.mark.parametrize("spec,dt", [
    ("cast:bf16;add;exp;cast:f32", F.F32),
    ("mul;cast:bf16;sigmoid", F.F16),
    ("add;mul;add;relu;scale:0.25;add", F.BF16),
])
def test_bf16_chains(spec, dt):
    n = 70_001
    inputs, _ = workloads.chain_inputs(spec, dt, n, 11)
    got, _ = _run_chain(spec, dt, inputs, (n,))
    _check(spec, dt, inputs, (n,), got)


@pytest.mark.parametrize("n", workloads.FLAT_SIZES)
@pytest.mark.parametrize("length", [1, 8, 32])
def test_flat_chain_full_sizes_sampled(n, length):
    """Full workload sizes; the oracle checks a sample (first/last elements,
    the ragged end, and random positions)."""
    spec, dt = workloads.random_chain(length, 5)
    c = F.fuse_compile(spec, (n,), dt)
    dev = [workloads.device_uniform(n, -2.0, 2.0, 1000 * j + length, d)
           for j, d in enumerate(c.in_dtypes)]
    out = Guarded(n, c.out_dtype)
    F.fuse_launch(c, dev, out.t)
    torch.cuda.synchronize()
    assert out.canary_ok()
    g = np.random.default_rng(n + length)
    idx = np.unique(np.concatenate([np.arange(min(n, 4096)), np.arange(max(0, n - 4096), n),
                                    g.integers(0, n, 200_000)]))
    it = torch.from_numpy(idx).cuda()
    ins = [to_host(t[it], d) for t, d in zip(dev, c.in_dtypes)]
    got = to_host(out.t[it], c.out_dtype)
    _check(spec, dt, ins, (len(idx),), got)


# ------------------------------------------------------------ shape buckets

@pytest.mark.parametrize("spec,dt,shape,rows_list", [
    ("add;relu;scale:0.5", F.F32, ((1 << 16) + 123,), [1, 7, 1000, 4097, (1 << 16) + 123]),
    ("mul;sigmoid;cast:f16;add", F.F32, (300, 37), [1, 2, 299, 300]),
    ("shuffle:4;add;sigmoid", F.F16, (8, 16, 7, 7), [1, 3, 8]),
    ("shuffle:2;exp;scale:0.25", F.F16, (6, 8, 4, 4), [1, 5, 6]),
])
def test_bucket_handle_runs_any_leading_dimension(spec, dt, shape, rows_list):
    c = F.fuse_compile_bucket(spec, shape, dt)
    inner = int(np.prod(shape[1:]))
    full = int(np.prod(shape))
    inputs, _ = workloads.chain_inputs(spec, dt, full, 31)
    dev = [to_dev(a, d) for a, d in zip(inputs, c.in_dtypes)]
    for rows in rows_list:
        n = rows * inner
        out = Guarded(n, c.out_dtype)
        F.fuse_launch_rows(c, dev, out.t, rows)
        torch.cuda.synchronize()
        assert out.canary_ok()
        sub = (rows,) + tuple(shape[1:])
        _check(spec, dt, [a[:n] for a in inputs], sub, to_host(out.t, c.out_dtype))


# ------------------------------------------------------------ ChannelShuffle prologue

@pytest.mark.parametrize("shape,groups", [
    ((2, 8, 4, 4), 4), ((1, 12, 3, 5), 3), ((3, 6, 1, 1), 2), ((2, 16, 8, 8), 16),
    ((2, 16, 8, 8), 1), ((1, 4, 7, 9), 2),
])
@pytest.mark.parametrize("length", [0, 1, 4])
def test_shuffle_chain_small(shape, groups, length):
    body, dt = workloads.random_chain(length, groups, start_dtype=F.F16) if length else ("", F.F16)
    spec = f"shuffle:{groups};" + body
    n = int(np.prod(shape))
    inputs, _ = workloads.chain_inputs(spec, dt, n, 3)
    got, _ = _run_chain(spec, dt, inputs, shape)
    if length == 0:
        assert np.array_equal(got, oracle.channel_shuffle(inputs[0].reshape(shape), groups)
                              .reshape(-1))
    else:
        _check(spec, dt, inputs, shape, got)


@pytest.mark.parametrize("length", workloads.CHAIN_LENGTHS)
def test_shuffle_chain_full_config(length):
    cfg = workloads.SHUFFLE_CHAIN
    body, dt = workloads.random_chain(length, 9, start_dtype=F.F16)
    spec = f"shuffle:{cfg['groups']};{body}"
    n = int(np.prod(cfg["shape"]))
    inputs, _ = workloads.chain_inputs(spec, dt, n, cfg["seed"])
    got, _ = _run_chain(spec, dt, inputs, cfg["shape"])
    _check(spec, dt, inputs, cfg["shape"], got)


# ------------------------------------------------------------ channel_shuffle entry point

@pytest.mark.parametrize("shape,groups,dt", [
    ((32, 256, 56, 56), 4, F.F16), ((2, 24, 5, 7), 3, F.F16), ((4, 8, 16, 16), 2, F.F32),
    ((1, 64, 9, 9), 8, F.BF16), ((2, 6, 1, 1), 6, F.F16), ((3, 16, 4, 4), 1, F.F16),
])
def test_channel_shuffle_bit_exact(shape, groups, dt):
    x = workloads.uniform(shape, -2, 2, 17, dt)
    xd = to_dev(x.reshape(-1), dt)
    out = Guarded(x.size, dt)
    F.channel_shuffle(xd, out.t, groups, dt, shape=shape)
    torch.cuda.synchronize()
    assert out.canary_ok()
    want = oracle.channel_shuffle(x, groups).reshape(-1)
    assert np.array_equal(to_host(out.t, dt), want)
    # round trip with the inverse group count
    back = Guarded(x.size, dt)
    F.channel_shuffle(out.t, back.t, shape[1] // groups, dt, shape=shape)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(back.t, dt), x.reshape(-1))


def test_channel_shuffle_unaligned():
    shape, groups, dt = (2, 8, 6, 6), 4, F.F16
    x = workloads.uniform(shape, -2, 2, 18, dt)
    xd = misaligned_copy(to_dev(x.reshape(-1), dt), 1)
    out = Guarded(x.size, dt, offset_elems=3)
    F.channel_shuffle(xd, out.t, groups, dt, shape=shape)
    torch.cuda.synchronize()
    assert out.canary_ok()
    assert np.array_equal(to_host(out.t, dt), oracle.channel_shuffle(x, groups).reshape(-1))


def test_empty_chain_is_noop():
    c = F.fuse_compile("add;relu", [0], F.F32)
    F.fuse_launch(c, [0, 0], 0)
    torch.cuda.synchronize()


def test_launch_count_is_one_per_chain():
    spec, dt = workloads.random_chain(16, 1)
    n = 1 << 20
    c = F.fuse_compile(spec, (n,), dt)
    dev = [workloads.device_uniform(n, -2, 2, j, d) for j, d in enumerate(c.in_dtypes)]
    out = torch.empty(n, dtype={0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[c.out_dtype],
                      device="cuda")
    before = F.fuse_stats()
    for _ in range(5):
        F.fuse_launch(c, dev, out)
    after = F.fuse_stats()
    assert after["launches"] - before["launches"] == 5
    assert after["compiles"] == before["compiles"]


# ------------------------------------------------------------ debug bounds checks

@pytest.mark.parametrize("spec,dt,shape,offset", [
    ("add;relu;scale:0.5", F.F32, ((1 << 20) + 7,), 0),   # vector chunks, remainder, tail
    ("mul;exp;cast:f16", F.F32, (4099,), 1),              # scalar kernel (misaligned)
    ("shuffle:4;sigmoid;add", F.F16, (2, 16, 8, 8), 0),   # shuffled vectors
    ("shuffle:3;relu", F.F16, (1, 12, 3, 5), 0),          # shuffled, scalar (HW % VEC != 0)
])
def test_debug_bounds_build_matches_and_reports_nothing(monkeypatch, spec, dt, shape, offset):
    # FUSE_DEBUG_BOUNDS=1 compiles an index check before every load and
    # store; on correct launches the results are unchanged and the device
    # error word stays 0
    monkeypatch.setenv("FUSE_DEBUG_BOUNDS", "1")
    assert "in_bounds(" in F.fuse_source(spec, shape, dt)
    n = int(np.prod(shape))
    inputs, _ = workloads.chain_inputs(spec, dt, n, 41)
    F.fuse_device_error()  # clear
    got, _ = _run_chain(spec, dt, inputs, shape, offset=offset)
    assert F.fuse_device_error() == 0
    _check(spec, dt, inputs, shape, got)


def test_debug_bounds_bucket_launch(monkeypatch):
    monkeypatch.setenv("FUSE_DEBUG_BOUNDS", "1")
    spec, dt, shape = "shuffle:4;add;sigmoid", F.F16, (8, 16, 7, 7)
    c = F.fuse_compile_bucket(spec, shape, dt)
    inner, full = int(np.prod(shape[1:])), int(np.prod(shape))
    inputs, _ = workloads.chain_inputs(spec, dt, full, 43)
    dev = [to_dev(a, d) for a, d in zip(inputs, c.in_dtypes)]
    F.fuse_device_error()
    for rows in (1, 3, 8):
        n = rows * inner
        out = Guarded(n, c.out_dtype)
        F.fuse_launch_rows(c, dev, out.t, rows)
        torch.cuda.synchronize()
        assert out.canary_ok() and F.fuse_device_error() == 0
        _check(spec, dt, [a[:n] for a in inputs], (rows,) + shape[1:], to_host(out.t, c.out_dtype))


# ------------------------------------------------------------ past 2^31 elements

def _big_sample(n, seed):
    # first and last elements, both sides of element 2^31, random positions;
    # every index checked on the host to lie inside the tensor
    g = np.random.default_rng(seed)
    edge = 1 << 31
    idx = np.unique(np.concatenate([np.arange(4096), np.arange(edge - 2048, min(edge + 2048, n)),
                                    np.arange(n - 4096, n), g.integers(0, n, 100_000)]))
    assert idx[0] >= 0 and idx[-1] < n
    return idx


def test_chain_past_2_to_the_31_elements():
    # 64-bit index arithmetic (2^31 + 13 fp16 elements, 3 tensors of 4.3 GB)
    if torch.cuda.mem_get_info()[0] < (40 << 30):
        pytest.skip("needs 40 GB of free device memory")
    n = (1 << 31) + 13
    spec, dt = "add;relu;scale:0.5", F.F16
    c = F.fuse_compile(spec, (n,), dt)
    assert "typedef long long idx_t;" in F.fuse_source(spec, (n,), dt)
    dev = [workloads.device_uniform(n, -2.0, 2.0, 77 + j, dt) for j in range(2)]
    out = Guarded(n, dt)
    F.fuse_launch(c, dev, out.t)
    torch.cuda.synchronize()
    assert out.canary_ok()
    idx = _big_sample(n, 78)
    it = torch.from_numpy(idx).cuda()
    ins = [to_host(t[it], dt) for t in dev]
    _check(spec, dt, ins, (len(idx),), to_host(out.t[it], dt))
    del dev, out


def test_shuffled_chain_past_2_to_the_31_elements():
    # the shuffle's plane index in 64-bit arithmetic: [2676, 256, 56, 56] fp16
    if torch.cuda.mem_get_info()[0] < (40 << 30):
        pytest.skip("needs 40 GB of free device memory")
    shape = (2676, 256, 56, 56)
    n = int(np.prod(shape))
    assert n > (1 << 31)
    spec, dt = "shuffle:4;sigmoid", F.F16
    c = F.fuse_compile(spec, shape, dt)
    x = workloads.device_uniform(n, -2.0, 2.0, 79, dt)
    out = Guarded(n, dt)
    F.fuse_launch(c, [x], out.t)
    torch.cuda.synchronize()
    assert out.canary_ok()
    idx = _big_sample(n, 80)
    got = to_host(out.t[torch.from_numpy(idx).cuda()], dt)
    host_x = to_host(x, dt)  # the oracle evaluates the sampled outputs from the whole input
    del x
    _check(spec, dt, [host_x], shape, got, idx=idx)


# ------------------------------------------------------------ output over an input

@pytest.mark.parametrize("over", [0, 2])
@pytest.mark.parametrize("offset", [0, 1])
def test_output_written_over_an_input(over, offset):
    """fuse.h allows the output to be the same pointer as an input of its
    dtype: every element is read before the thread that owns it writes it."""
    spec, dt, n = "add;mul;relu;sigmoid;scale:0.75", F.F32, 10_007
    inputs, _ = workloads.chain_inputs(spec, dt, n, 60 + over)
    c = F.fuse_compile(spec, (n,), dt)
    dev = [to_dev(a, d) for a, d in zip(inputs, c.in_dtypes)]
    if offset:
        dev = [misaligned_copy(t, offset) for t in dev]
    F.fuse_launch(c, dev, dev[over])
    torch.cuda.synchronize()
    got = to_host(dev[over], c.out_dtype)
    fails, counts, _ = oracle.chain_check(spec, dt, inputs, (n,), got)
    assert fails == 0 and counts[3] == 0, counts
    # the other inputs are untouched
    for j, (t, a) in enumerate(zip(dev, inputs)):
        if j != over:
            assert np.array_equal(to_host(t, c.in_dtypes[j]), a)


# ------------------------------------------------------------ configuration fuzz

@pytest.mark.parametrize("block", range(6))
def test_random_configurations(block):
    """Seeded random chains over the planner's whole range: 1-32 ops, start
    dtype f16, f32 or bf16, sizes from 1 to ~300k elements, a shuffle prefix on
    random NCHW shapes, and unaligned pointers (the scalar kernel).  Every case
    against the oracle."""
    rng = np.random.default_rng(7000 + block)
    for _ in range(25):
        length = int(rng.integers(1, 33))
        seed = int(rng.integers(0, 1_000_000))
        start = (F.F16, F.F32, F.BF16)[int(rng.integers(0, 3))]
        spec, dt = workloads.random_chain(length, seed, start_dtype=start)
        if rng.random() < 0.3:
            groups = int(rng.choice([1, 2, 4, 8]))
            shape = (int(rng.integers(1, 4)), groups * int(rng.integers(1, 9)),
                     int(rng.integers(1, 12)), int(rng.integers(1, 12)))
            spec = f"shuffle:{groups};{spec}"
        else:
            shape = (int(rng.choice([1, 7, 31, 255, 4097, 65_543, int(rng.integers(1, 300_000))])),)
        offset = int(rng.random() < 0.25)
        n = int(np.prod(shape))
        inputs, _ = workloads.chain_inputs(spec, dt, n, seed)
        got, _ = _run_chain(spec, dt, inputs, shape, offset)
        _check(spec, dt, inputs, shape, got)
