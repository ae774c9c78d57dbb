"""The C ABI from a plain C program (tests/c_abi/chain_demo.c): built with gcc
against include/fuse.h and libfusechain.so.  Without a GPU the program must
compile a chain and report that there is no device; on a GPU it must
produce add -> relu -> scale bit-exactly."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.join(ROOT, "elementwise_chain_jit_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    exe = str(tmp_path / "chain_demo")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", os.path.join(HERE, "c_abi", "chain_demo.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", PKG, "-lfusechain", f"-Wl,-rpath,{PKG}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe):
    return subprocess.run([exe], capture_output=True, text=True, timeout=300)


def test_c_program_builds_and_compiles_a_chain(tmp_path):
    r = _run(_build(tmp_path))
    assert r.returncode == 0, (r.stdout, r.stderr)
    assert r.stdout.startswith("compiled; no CUDA device") or r.stdout.startswith("ok:")


@pytest.mark.gpu
def test_c_program_runs_the_chain_bit_exactly(tmp_path):
    r = _run(_build(tmp_path))
    assert r.returncode == 0, (r.stdout, r.stderr)
    assert r.stdout.startswith("ok: 0 of 1048583 elements differ, 1 launch"), r.stdout
