"""GPU parity of rmsnorm_linear (RMSNorm -> Linear -> scale on tcgen05) against
the oracle, through the C ABI.  Tolerances (tests/tolerance.py): bf16 outputs
within 8e-3 relative to the sum of the magnitudes of the dot product's terms;
fp16 outputs within 2 ulp of the correctly rounded value, or a correct
rounding of a value within the derived bound of the computation (the product
w * gamma rounded to fp16, fp32 accumulation on the tensor cores).  Each case
also checks that no bounded wait inside the kernel ran out."""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads
import tolerance as tol
from gpu_util import Guarded, to_dev, to_host

pytestmark = pytest.mark.gpu


def _check(got, dt, x, want, mag, scale, K, eps=1e-6, what="rmsnorm_linear"):
    """got: device storage [rows, N]; x: the rows' inputs [rows, K] storage."""
    xd = oracle.to_double(x, dt)
    s = 1.0 / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps)
    sx = abs(scale) * s * np.abs(xd).sum(axis=1, keepdims=True)
    tol.assert_accepted(got, dt, want, mag, tol.contraction_bound(mag, dt, K, sx), what=what)


def _case(M, N, K, dt, seed, bias=True, scale=0.75, rows=None):
    x = workloads.normal((M, K), 0, 1, seed, dt)
    g = workloads.normal(K, 1, 0.1, seed + 1, dt)
    w = workloads.normal((N, K), 0, 1 / np.sqrt(K), seed + 2, dt)
    b = workloads.normal(N, 0, 0.5, seed + 3, dt) if bias else None
    out = Guarded(M * N, dt)
    F.rmsnorm_linear(to_dev(x.reshape(-1), dt), to_dev(g, dt), to_dev(w.reshape(-1), dt),
                     None if b is None else to_dev(b, dt), out.t, 1e-6, scale, dt, M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert F.fuse_device_error() == 0
    assert out.canary_ok()
    sel = np.arange(M) if rows is None else np.asarray(rows)
    want, mag = oracle.rmsnorm_linear(x, g, w, b, dt, 1e-6, scale, rows=sel)
    _check(to_host(out.t, dt).reshape(M, N)[sel], dt, x[sel], want, mag, scale, K)


def test_tiny_one_tile_one_k_step():
    _case(128, 256, 64, F.BF16, 1)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (256, 512, 256), (384, 768, 1024)])
@pytest.mark.parametrize("dt", [F.BF16, F.F16])
def test_small_shapes(M, N, K, dt):
    _case(M, N, K, dt, 10 + K % 97)


def test_no_bias_and_negative_scale():
    _case(256, 256, 320, F.BF16, 20, bias=False, scale=-1.5)


def test_full_size_sampled_rows():
    M, N, K = 16384, 4096, 4096
    _case(M, N, K, F.BF16, 30, rows=[0, 1, 127, 128, 5000, 16383])


def test_rejects_unsupported_shapes_and_dtypes():
    for g in (256, None):  # both paths: TMA row strides of 16 bytes
        for N, K in ((260, 64), (256, 60), (256, 0)):
            with pytest.raises(F.FuseError) as e:
                F.rmsnorm_linear(256, g, 256, 256, 256, 1e-6, 1.0, F.BF16, M=128, N=N, K=K)
            assert e.value.code == -2
        # TMA row coordinates are 32-bit
        with pytest.raises(F.FuseError) as e:
            F.rmsnorm_linear(256, g, 256, 256, 256, 1e-6, 1.0, F.BF16, M=2 ** 31, N=256, K=64)
        assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.rmsnorm_linear(256, 256, 256, 256, 256, 1e-6, 1.0, F.F32, M=128, N=256, K=64)
    assert e.value.code == -3


def _folded_case(M, N, K, dt, seed, rows=None, bias=True):
    x = workloads.normal((M, K), 0, 1, seed, dt)
    g = workloads.normal(K, 1, 0.1, seed + 1, dt)
    w = workloads.normal((N, K), 0, 1 / np.sqrt(K), seed + 2, dt)
    b = workloads.normal(N, 0, 0.5, seed + 3, dt) if bias else None
    wd = to_dev(w.reshape(-1), dt)
    wf = torch.empty_like(wd)
    F.rmsnorm_linear_fold(wd, to_dev(g, dt), wf, dt, N=N, K=K)
    out = Guarded(M * N, dt)
    F.rmsnorm_linear(to_dev(x.reshape(-1), dt), None, wf, None if b is None else to_dev(b, dt),
                     out.t, 1e-6, 0.5, dt, M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert F.fuse_device_error() == 0
    assert out.canary_ok()
    # the folded weight is w * gamma rounded once
    assert np.array_equal(to_host(wf, dt).reshape(N, K),
                          oracle.store(oracle.to_double(w, dt) * oracle.to_double(g, dt), dt))
    sel = np.arange(M) if rows is None else np.asarray(rows)
    want, mag = oracle.rmsnorm_linear(x, g, w, b, dt, 1e-6, 0.5, rows=sel)
    _check(to_host(out.t, dt).reshape(M, N)[sel], dt, x[sel], want, mag, 0.5, K)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (384, 256, 448), (640, 768, 128)])
@pytest.mark.parametrize("dt", [F.BF16, F.F16])
def test_folded_gamma_fast_path(M, N, K, dt):
    _folded_case(M, N, K, dt, 40 + K % 89)


def test_folded_full_size_sampled_rows():
    _folded_case(16384, 4096, 4096, F.BF16, 50, rows=[0, 3, 129, 8191, 16383])


@pytest.mark.parametrize("bias", [True, False])
def test_folded_many_tiles_per_cta(bias):
    # 80 x 8 = 640 output tiles on at most one CTA per SM: every CTA of the
    # persistent kernel takes several tiles, so both TMEM accumulator buffers
    # and both phases of their barriers are reused; every row is checked
    _folded_case(10240, 2048, 128, F.BF16, 60, bias=bias)


@pytest.mark.parametrize("M,N,K,dt", [(1, 8, 8, F.BF16), (50, 264, 72, F.BF16),
                                      (1000, 520, 200, F.F16), (130, 256, 4104, F.BF16)])
def test_folded_ragged_shapes(M, N, K, dt):
    # rows, columns and k-steps past the tensors: zeros on load, clipped on
    # store (the output's canaries catch a store past M * N)
    _folded_case(M, N, K, dt, 70 + M % 13)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (100, 264, 72), (300, 520, 200)])
def test_gamma_path_ragged_shapes(M, N, K):
    # gamma given: folded into a stream-ordered scratch copy of w for the call,
    # so the gamma path takes the same shapes as the folded one
    _case(M, N, K, F.BF16, 90 + M % 11)


def test_gamma_path_on_two_streams_at_once():
    # two calls with different gamma on two streams: each folds into its own
    # scratch copy of w, taken from and returned to its stream's pool
    M, N, K, dt = 512, 512, 256, F.BF16
    x = workloads.normal((M, K), 0, 1, 95, dt)
    w = workloads.normal((N, K), 0, 1 / np.sqrt(K), 96, dt)
    gs = [workloads.normal(K, 1, 0.1, 97 + i, dt) for i in range(2)]
    xd, wd = to_dev(x.reshape(-1), dt), to_dev(w.reshape(-1), dt)
    gd = [to_dev(g, dt) for g in gs]
    outs = [torch.empty(M * N, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(3):
        for i in range(2):
            F.rmsnorm_linear(xd, gd[i], wd, None, outs[i], 1e-6, 1.0, dt, M=M, N=N, K=K,
                             stream=streams[i])
    torch.cuda.synchronize()
    assert F.fuse_device_error() == 0
    for i in range(2):
        want, mag = oracle.rmsnorm_linear(x, gs[i], w, None, dt, 1e-6, 1.0)
        _check(to_host(outs[i], dt).reshape(M, N), dt, x, want, mag, 1.0, K)


def test_mixed_run_schedule_every_row():
    """16384 x 4096 on the GPU's clusters deals runs of 4 column blocks for most
    row pairs and runs of 2 for the last ones: every row is checked, on columns
    from each of the 16 column blocks (an output column depends only on its
    row of w, so the oracle takes just those rows of w)."""
    M, N, K, dt = 16384, 4096, 64, F.BF16
    x = workloads.normal((M, K), 0, 1, 90, dt)
    g = workloads.normal(K, 1, 0.1, 91, dt)
    w = workloads.normal((N, K), 0, 1 / np.sqrt(K), 92, dt)
    b = workloads.normal(N, 0, 0.5, 93, dt)
    out = torch.empty(M * N, dtype=torch.bfloat16, device="cuda")
    F.rmsnorm_linear(to_dev(x.reshape(-1), dt), to_dev(g, dt), to_dev(w.reshape(-1), dt),
                     to_dev(b, dt), out, 1e-6, 0.5, dt, M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert F.fuse_device_error() == 0
    cols = np.unique(np.concatenate([np.arange(0, N, 256), np.arange(255, N, 256),
                                     np.random.default_rng(9).integers(0, N, 32)]))
    want, mag = oracle.rmsnorm_linear(x, g, w[cols], b[cols], dt, 1e-6, 0.5)
    _check(to_host(out.view(M, N)[:, torch.from_numpy(cols).cuda()], dt), dt, x, want, mag, 0.5, K)


@pytest.mark.parametrize("block", range(3))
def test_random_shapes(block):
    """Seeded random shapes on both paths: any M, N and K multiples of 8 (one
    to several row tiles, column blocks and k-steps with ragged edges), both
    dtypes, with and without bias."""
    rng = np.random.default_rng(500 + block)
    for i in range(8):
        M = int(rng.integers(1, 701))
        N = 8 * int(rng.integers(1, 129))
        K = 8 * int(rng.integers(1, 129))
        dt = (F.BF16, F.F16)[int(rng.integers(0, 2))]
        bias = bool(rng.random() < 0.7)
        if rng.random() < 0.5:
            _case(M, N, K, dt, 600 + 10 * block + i, bias=bias)
        else:
            _folded_case(M, N, K, dt, 700 + 10 * block + i, bias=bias)
