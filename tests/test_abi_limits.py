"""Every size limit include/fuse.h documents, called just inside and just
outside, through the C ABI.

Just outside, the call must fail with the documented status before any
device work.  Just inside, the call must get past validation: on a machine
with no GPU it then fails at the first device step with FUSE_E_CUDA (the
kernel is generated and compiled first), which shows the limit is where the
header puts it.  The pointers are placeholders that are never dereferenced,
so the inside calls run only where there is no GPU.
"""
import pytest
import torch

import elementwise_chain_jit_gb300 as F

NO_GPU = not torch.cuda.is_available()
P = 256  # placeholder device address (16-byte aligned), never dereferenced
E_SPEC, E_SHAPE, E_DTYPE, E_ARG, E_CUDA = -1, -2, -3, -8, -7


def outside(call, code):
    with pytest.raises(F.FuseError) as e:
        call()
    assert e.value.code == code, (e.value.code, str(e.value))


def inside(call):
    if not NO_GPU:
        pytest.skip("the inside calls use placeholder pointers: run where no GPU is visible")
    with pytest.raises(F.FuseError) as e:
        call()
    assert e.value.code == E_CUDA, (e.value.code, str(e.value))


def test_chain_dims_and_element_count():
    # 1..8 dims; up to 2^40 elements (compiling needs no device)
    F.fuse_compile("relu", [2] * 8, F.F32)
    outside(lambda: F.fuse_compile("relu", [2] * 9, F.F32), E_SHAPE)
    F.fuse_compile("relu", [1 << 20, 1 << 20], F.F16)
    outside(lambda: F.fuse_compile("relu", [(1 << 20) + 1, 1 << 20], F.F16), E_SHAPE)


def test_chain_op_and_input_counts():
    F.fuse_compile(";".join(["relu"] * 1024), [64], F.F32)
    outside(lambda: F.fuse_compile(";".join(["relu"] * 1025), [64], F.F32), E_SPEC)
    c = F.fuse_compile(";".join(["add"] * 127), [64], F.F32)  # 128 input tensors
    assert c.n_in == 128
    outside(lambda: F.fuse_compile(";".join(["add"] * 128), [64], F.F32), E_SPEC)


def test_shuffle_groups():
    F.fuse_compile("shuffle:1;relu", [1, 4, 2, 2], F.F16)
    F.fuse_compile(f"shuffle:{1 << 20};relu", [1, 1 << 20, 1, 1], F.F16)
    outside(lambda: F.fuse_compile("shuffle:0;relu", [1, 4, 2, 2], F.F16), E_SPEC)
    outside(lambda: F.fuse_compile(f"shuffle:{(1 << 20) + 1};relu", [1, 4, 2, 2], F.F16), E_SPEC)
    outside(lambda: F.fuse_compile("shuffle:3;relu", [1, 4, 2, 2], F.F16), E_SHAPE)


def test_bucket_rows():
    b = F.fuse_compile_bucket("add", [64, 3], F.F32)
    outside(lambda: F.fuse_launch_rows(b, [P, P], P, 65, stream=0), E_SHAPE)
    outside(lambda: F.fuse_launch_rows(b, [P, P], P, -1, stream=0), E_SHAPE)
    inside(lambda: F.fuse_launch_rows(b, [P, P], P, 64, stream=0))


@pytest.mark.parametrize("fn", ["rmsnorm", "layernorm"])
def test_norm_row_length(fn):
    def call(hidden, rows=4, eps=1e-6):
        if fn == "rmsnorm":
            return lambda: F.rmsnorm_residual(P, P, P, P, P, eps, F.BF16, rows=rows,
                                              hidden=hidden, stream=0)
        return lambda: F.layernorm_residual(P, P, P, P, P, P, eps, F.BF16, rows=rows,
                                            hidden=hidden, stream=0)
    outside(call(0), E_SHAPE)
    outside(call(65537), E_SHAPE)
    outside(call(64, rows=-1), E_SHAPE)
    outside(call(64, eps=-1e-30), E_ARG)
    inside(call(1))
    inside(call(65536))
    inside(call(64, eps=0.0))


def test_layernorm_residual_pairing():
    outside(lambda: F.layernorm_residual(P, P, P, P, P, None, 1e-5, F.BF16, rows=4, hidden=64,
                                         stream=0), E_ARG)


def test_rmsnorm_linear_shapes():
    def call(M=128, N=256, K=64, dt=F.BF16, gamma=None):
        return lambda: F.rmsnorm_linear(P, gamma, P, P, P, 1e-6, 1.0, dt, M=M, N=N, K=K,
                                        stream=0)
    outside(call(dt=F.F32), E_DTYPE)
    outside(call(N=260), E_SHAPE)
    outside(call(K=60), E_SHAPE)
    outside(call(K=0), E_SHAPE)
    outside(call(K=(1 << 20) + 8), E_SHAPE)
    outside(call(M=(1 << 31) - 128), E_SHAPE)
    inside(call(M=(1 << 31) - 129))
    inside(call(K=1 << 20, M=128))
    outside(lambda: F.rmsnorm_linear_fold(P, P, P, F.BF16, N=256, K=(1 << 20) + 1, stream=0),
            E_SHAPE)
    outside(lambda: F.rmsnorm_linear_fold(P, P, P, F.BF16, N=256, K=0, stream=0), E_SHAPE)


@pytest.mark.parametrize("noalloc", [False, True])
def test_rope_shapes_and_positions(noalloc):
    fn = F.rope_qkv_split_noalloc if noalloc else F.rope_qkv_split

    def call(tokens=4, heads=2, hd=64, pos0=0, base=10000.0):
        return lambda: fn(P, P, P, P, heads, hd, pos0, base, F.BF16, tokens=tokens, stream=0)
    outside(call(hd=0), E_SHAPE)
    outside(call(hd=1026), E_SHAPE)
    outside(call(hd=63), E_SHAPE)
    outside(call(heads=0), E_SHAPE)
    outside(call(heads=1025, hd=1024), E_SHAPE)  # heads * head_dim <= 2^20
    outside(call(heads=(1 << 30), hd=1024), E_SHAPE)
    outside(call(tokens=-1), E_SHAPE)
    # every position below 2^22: pos0 + tokens <= 2^22
    outside(call(tokens=4, pos0=(1 << 22) - 3), E_SHAPE)
    outside(call(tokens=0, pos0=(1 << 22) + 1), E_SHAPE)
    outside(call(pos0=-1), E_SHAPE)
    outside(call(base=1.0), E_ARG)
    outside(call(base=float("inf")), E_ARG)
    # products that would overflow 64 bits are refused, not wrapped
    outside(call(tokens=1 << 62, hd=1024), E_SHAPE)
    outside(call(tokens=1, pos0=(1 << 63) - 1), E_SHAPE)
    inside(call(tokens=4, pos0=(1 << 22) - 4))
    inside(call(hd=1024, tokens=2))
    inside(call(heads=1024, hd=1024, tokens=2))
    inside(call(hd=2))
    if noalloc:
        # its fixed array: tokens * head_dim <= 2^20
        outside(call(tokens=(1 << 13) + 1, hd=128), E_SHAPE)
        inside(call(tokens=1 << 13, hd=128))
    else:
        outside(call(tokens=1 << 31, pos0=0), E_SHAPE)


def test_detect_counts_and_sizes():
    def call(hw=((4, 4),), na=3, no=85):
        ns = len(hw)
        return lambda: F.detect_decode([P] * ns, list(hw), [8.0 * (s + 1) for s in range(ns)],
                                       [[[1.0, 2.0]] * na] * ns, na, no, P, F.F16, stream=0)
    outside(call(hw=()), E_SHAPE)
    outside(call(hw=((2, 2),) * 9), E_SHAPE)
    outside(call(na=0), E_SHAPE)
    outside(call(na=17), E_SHAPE)
    outside(call(no=4), E_SHAPE)
    outside(call(no=1025), E_SHAPE)
    outside(call(hw=((1 << 12, (1 << 12) + 1),)), E_SHAPE)  # H*W <= 2^24
    outside(call(hw=((0, 4),)), E_SHAPE)
    inside(call(hw=((2, 2),) * 8, na=16, no=5))
    inside(call(no=1024, na=1))
    inside(call(hw=((1 << 12, 1 << 12),), na=1, no=5))


def test_channel_shuffle_arguments():
    def call(shape=(2, 16, 8, 8), groups=4, out=2 * P):
        return lambda: F.channel_shuffle(P, out, groups, F.F16, shape=shape, stream=0)
    outside(call(groups=0), E_ARG)
    outside(call(groups=3), E_SHAPE)
    outside(call(out=P), E_ARG)  # in place
    outside(call(shape=(2, -16, 8, 8)), E_SHAPE)
    outside(call(shape=((1 << 24) + 1, 16, 64, 64)), E_SHAPE)  # above 2^40 elements
    outside(call(shape=(1, 1 << 40, 1 << 40, 1 << 40), groups=1), E_SHAPE)  # no wrap-around
    inside(call(shape=(1 << 24, 16, 64, 64)))  # exactly 2^40 elements
    inside(call(shape=(3, 16, 8, 24)))


def test_selftest_spins():
    outside(lambda: F.fuse_selftest_bounded_wait(0, stream=0), E_ARG)
    outside(lambda: F.fuse_selftest_bounded_wait((1 << 30) + 1, stream=0), E_ARG)
    inside(lambda: F.fuse_selftest_bounded_wait(1 << 30, stream=0))
