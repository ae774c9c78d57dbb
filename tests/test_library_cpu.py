"""Host-side tests of the library that need no GPU.

  * the shared library loads and exports every symbol include/fuse.h declares;
  * spec parsing and validation errors come back as status codes + messages;
  * the generated sources bake the sizes, vector width and tail in;
  * every kernel family compiles with NVRTC for sm_103a, without spills;
  * calls that need a device fail cleanly (FUSE_E_CUDA) when there is none.
"""
import os
import re
import subprocess

import pytest
import torch

import elementwise_chain_jit_gb300 as F

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fuse.h")
NO_GPU = not torch.cuda.is_available()


def test_exports_every_declared_symbol():
    text = open(HEADER).read()
    declared = set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\(", text, re.M))
    assert declared == set(F.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines()}
    missing = declared - exported
    assert not missing, missing


@pytest.mark.parametrize("spec,code", [
    ("add;frobnicate", -1), ("scale:abc", -1), ("scale:inf", -1), ("relu:3", -1),
    ("cast:f64", -1), ("add;shuffle:2", -1), ("shuffle:0", -1), ("shuffle:x;relu", -1),
])
def test_bad_specs(spec, code):
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile(spec, [64], F.F32)
    assert e.value.code == code
    assert F.fuse_last_error()


def test_bad_shapes_and_dtypes():
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("shuffle:3;relu", [2, 8, 4, 4], F.F16)  # 8 % 3
    assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("shuffle:2;relu", [2, 8, 16], F.F16)  # not NCHW
    assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("relu", [-1], F.F16)
    assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("relu", [1 << 21, 1 << 20], F.F16)  # 2^41 elements
    assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("relu", [16], 7)
    assert e.value.code == -3


def test_chain_typing():
    c = F.fuse_compile("add;cast:f32;mul;cast:bf16;add", [1000], F.F16)
    assert c.n_in == 4
    assert c.in_dtypes == [F.F16, F.F16, F.F32, F.BF16]
    assert c.out_dtype == F.BF16


def test_source_bakes_sizes_vector_and_tail():
    src = F.fuse_source("add;relu;scale:0.5", [(1 << 26) + 7], F.F32)
    assert "constexpr long long N = 67108871LL;" in src
    assert "constexpr int VEC = 8;" in src  # 32 bytes of fp32
    assert "constexpr int TAIL = (int)(N - NVEC * VEC);" in src
    # a small tensor gets smaller chunks (about 8 CTAs per SM): 16-byte
    # vectors, one per thread, 128-thread CTAs
    small = F.fuse_source("add;relu;scale:0.5", [(1 << 20) + 7], F.F32)
    assert "constexpr int VEC = 4;" in small and "constexpr int BLOCK = 128;" in small
    assert "constexpr int UNROLL = 1;" in small
    assert "x = x * 0x1p-1f;" in src       # the scale constant, exact
    assert "x = x > 0.f ? x : 0.f;" in src
    assert "fuse_chain_vec" in src and "fuse_chain_scalar" in src
    src16 = F.fuse_source("relu", [1 << 26], F.F16)
    assert "constexpr int VEC = 16;" in src16  # 32 bytes of fp16
    shf = F.fuse_source("shuffle:4;relu", [32, 256, 56, 56], F.F16)
    assert "G = 4" in shf and "src_vec" in shf and "HW = 3136" in shf


def test_bucket_helper_and_source():
    assert [F.fuse_bucket(n) for n in (0, 1, 2, 3, 5, 1000, 1024, 1025)] == \
        [1, 1, 2, 4, 8, 1024, 1024, 2048]
    src = F.fuse_source_bucket("shuffle:4;add;sigmoid", [8, 16, 7, 7], F.F16)
    assert "long long n; };" in src and "#define SIZE_N(a) ((a).n)" in src
    fixed = F.fuse_source("shuffle:4;add;sigmoid", [8, 16, 7, 7], F.F16)
    assert "#define SIZE_N(a) N" in fixed


def test_launch_rows_checks_the_leading_dimension():
    fixed = F.fuse_compile("add;relu", [64, 3], F.F32)
    with pytest.raises(F.FuseError) as e:
        F.fuse_launch_rows(fixed, [256, 256], 256, 32, stream=0)
    assert e.value.code == -2  # a fixed handle runs only its own leading dimension
    bucket = F.fuse_compile_bucket("add;relu", [64, 3], F.F32)
    with pytest.raises(F.FuseError) as e:
        F.fuse_launch_rows(bucket, [256, 256], 256, 65, stream=0)
    assert e.value.code == -2  # above the bucket
    F.fuse_launch_rows(bucket, [0, 0], 0, 0, stream=0)  # nothing to do


def test_source_of_copy_and_odd_shuffle():
    # no ops: a bit copy; a plane size that is not a vector multiple: scalar only
    src = F.fuse_source("shuffle:2", [1, 4, 3, 3], F.F16)
    assert "copy" in src and "fuse_chain_vec" not in src


def _ptxas_log(monkeypatch, fn):
    monkeypatch.setenv("FUSE_PTXAS_VERBOSE", "1")
    fn()


@pytest.mark.skipif(not NO_GPU, reason="checks the no-device error path")
def test_fixed_entry_points_compile_then_report_no_device():
    before = F.fuse_stats()["compiles"]
    ptr = 256
    for call in (
        lambda: F.rmsnorm_residual(ptr, ptr, ptr, ptr, ptr, 1e-6, F.BF16, rows=16, hidden=4096,
                                   stream=0),
        lambda: F.layernorm_residual(ptr, ptr, ptr, ptr, ptr, ptr, 1e-5, F.BF16, rows=16,
                                     hidden=4096, stream=0),
        lambda: F.layernorm_residual(ptr, None, None, None, ptr, None, 1e-5, F.F32, rows=16,
                                     hidden=1000, stream=0),
        lambda: F.rope_qkv_split(ptr, ptr, ptr, ptr, 32, 128, 0, 10000.0, F.BF16, tokens=64,
                                 stream=0),
        lambda: F.detect_decode([ptr, ptr, ptr], [(8, 8), (4, 4), (2, 2)], [8, 16, 32],
                                [[[1, 2]] * 3] * 3, 3, 85, ptr, F.F16, stream=0),
        lambda: F.channel_shuffle(ptr, ptr * 2, 4, F.F16, shape=(2, 16, 8, 8), stream=0),
    ):
        with pytest.raises(F.FuseError) as e:
            call()
        assert e.value.code == -7 and "driver" in str(e.value)
    assert F.fuse_stats()["compiles"] >= before + 6  # codegen + NVRTC ran before the device step


def test_argument_validation():
    with pytest.raises(F.FuseError) as e:
        F.rmsnorm_residual(256, 256, 256, 256, 256, 1e-6, F.BF16, rows=4, hidden=0, stream=0)
    assert e.value.code == -2
    with pytest.raises(F.FuseError) as e:
        F.rmsnorm_residual(0, 256, 256, 256, 256, 1e-6, F.BF16, rows=4, hidden=64, stream=0)
    assert e.value.code == -4
    with pytest.raises(F.FuseError) as e:
        F.rope_qkv_split(256, 256, 256, 256, 4, 127, 0, 10000.0, F.BF16, tokens=4, stream=0)
    assert e.value.code == -2  # odd head_dim
    with pytest.raises(F.FuseError) as e:
        F.rope_qkv_split(256, 256, 256, 256, 4, 128, (1 << 22) - 1, 10000.0, F.BF16, tokens=4,
                         stream=0)
    assert e.value.code == -2  # positions beyond the table limit
    with pytest.raises(F.FuseError) as e:
        F.detect_decode([256], [(4, 4)], [8], [[[1, 2]]], 1, 3, 256, F.F16, stream=0)
    assert e.value.code == -2  # no < 5
    with pytest.raises(F.FuseError) as e:
        F.channel_shuffle(256, 256, 3, F.F16, shape=(2, 16, 8, 8), stream=0)
    assert e.value.code == -2  # 16 % 3
    with pytest.raises(F.FuseError) as e:  # row coordinates past 32 bits
        F.rmsnorm_linear(256, None, 256, 256, 256, 1e-6, 1.0, F.BF16, M=2 ** 31, N=256, K=64,
                         stream=0)
    assert e.value.code == -2
    # empty work is a no-op, even without a device
    F.rmsnorm_residual(0, 0, 0, 0, 0, 1e-6, F.BF16, rows=0, hidden=64, stream=0)
    F.rope_qkv_split(0, 0, 0, 0, 4, 128, 0, 10000.0, F.BF16, tokens=0, stream=0)
    c = F.fuse_compile("add;relu", [0], F.F32)
    F.fuse_launch(c, [0, 0], 0, stream=0)
    with pytest.raises(F.FuseError) as e:
        F.fuse_launch(c, [0], 0, stream=0)
    assert e.value.code == -8  # wrong input count


def _compile_log(monkeypatch, spec, shape, dt):
    return F.fuse_source(spec, shape, dt)


@pytest.mark.parametrize("spec,shape,dt", [
    ("add;relu;scale:0.5", [1 << 20], F.F32),
    ("shuffle:4;cast:f32;add;sigmoid;exp;mul;cast:f16", [32, 256, 56, 56], F.F16),
    (";".join(["add", "mul"] * 16), [(1 << 24) + 7], F.F32),
    (";".join(["sigmoid", "exp", "cast:f32", "cast:f16"] * 8), [(1 << 28) + 7], F.F16),
])
def test_chain_kernels_compile_without_spills(spec, shape, dt):
    env = dict(os.environ, FUSE_PTXAS_VERBOSE="1")
    code = ("import elementwise_chain_jit_gb300 as F\n"
            f"F.fuse_compile({spec!r}, {shape!r}, {dt})\n")
    r = subprocess.run(["python", "-c", code], env=env, capture_output=True, text=True,
                       cwd=os.path.dirname(os.path.dirname(__file__)))
    assert r.returncode == 0, r.stderr
    assert "fuse_chain_vec" in r.stderr or "shuffle" in spec
    spills = re.findall(r"(\d+) bytes spill stores", r.stderr)
    assert spills and all(s == "0" for s in spills), r.stderr


def test_debug_bounds_source(monkeypatch):
    spec, shape = "shuffle:4;add;sigmoid", (2, 16, 8, 8)
    assert "in_bounds(" not in F.fuse_source(spec, shape, F.F16)
    monkeypatch.setenv("FUSE_DEBUG_BOUNDS", "1")
    src = F.fuse_source(spec, shape, F.F16)
    assert "struct Args { const void* in[NIN]; void* out; long long n; int* err; };" in src
    assert src.count("in_bounds(a, v, nvec) || !in_bounds(a, src_vec(v), nvec)") == 2
    assert "in_bounds(a, e, SIZE_N(a)) || !in_bounds(a, src_elem(e), SIZE_N(a))" in src
    F.fuse_compile(spec, shape, F.F16)  # and it compiles


def test_empty_inputs_succeed_without_a_launch():
    # nothing to do is FUSE_OK before any device work: these pass on a box
    # with no GPU, and launch nothing
    before = F.fuse_stats()["launches"]
    F.rmsnorm_residual(256, 256, 256, 256, 256, 1e-6, F.BF16, rows=0, hidden=4096)
    F.layernorm_residual(256, 256, 256, 256, 256, 256, 1e-5, F.BF16, rows=0, hidden=4096)
    F.rope_qkv_split(256, 256, 256, 256, 32, 128, 0, 10000.0, F.BF16, tokens=0)
    F.rmsnorm_linear(256, None, 256, 256, 256, 1e-6, 1.0, F.BF16, M=0, N=256, K=64)
    c = F.fuse_compile("add;relu;scale:0.5", (0,), F.F32)
    F.fuse_launch(c, [256, 256], 256)
    F.channel_shuffle(256, 512, 4, F.F16, shape=(0, 8, 4, 4))
    assert F.fuse_stats()["launches"] == before


def test_detect_decoder_checks_the_feature_count():
    dec = F.DetectDecoder([(8, 8), (4, 4)], [8, 16], [[[1, 2]] * 3] * 2, 3, 85, F.F16)
    with pytest.raises(ValueError):
        dec([256], 256, stream=0)


@pytest.mark.skipif(not NO_GPU, reason="checks the no-device error path")
def test_bound_launch_reaches_the_device_step():
    c = F.fuse_compile("add;relu;scale:0.5", (1024,), F.F32)
    step = c.bind([256, 512], 768)
    with pytest.raises(F.FuseError) as e:
        step()
    assert e.value.code == -7  # validated, then no driver
    with pytest.raises(F.FuseError) as e:
        c.bind([256], 768)()   # one input where the chain takes two
    assert e.value.code == -8  # FUSE_E_ARG, before any device step
