"""The compile cache on disk and host-side fault injection (no GPU: NVRTC
compiles on the CPU).

  * a CUBIN written to FUSE_CACHE_DIR by one process is loaded by the next
    instead of being compiled again;
  * a damaged or truncated cache file is detected and recompiled, never
    handed to the driver;
  * a build of the library whose kernel headers differ keys its cache
    entries apart, so it never loads another build's CUBIN;
  * an unwritable cache directory is ignored;
  * an NVRTC failure forced through FUSE_NVRTC_OPTIONS returns FUSE_E_COMPILE
    with the compiler's log and leaves the library usable.
"""
import json
import os
import shutil
import subprocess
import sys

import pytest

import elementwise_chain_jit_gb300 as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SPEC = "add;sigmoid;scale:0.375;cast:f16"  # a chain no other test compiles

SCRIPT = """
import json, sys
sys.path.insert(0, {root!r})
import elementwise_chain_jit_gb300 as F
assert F.__file__.startswith({root!r}), F.__file__
F.fuse_compile({spec!r}, (4099,), F.F32)
print(json.dumps(F.fuse_stats()))
"""


def _run(cache_dir, root=ROOT):
    env = dict(os.environ, FUSE_CACHE_DIR=str(cache_dir))
    env.pop("FUSE_NVRTC_OPTIONS", None)
    out = subprocess.run([sys.executable, "-c", SCRIPT.format(root=root, spec=SPEC)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    return json.loads(out.stdout.strip().splitlines()[-1])


def _files(d):
    return sorted(p for p in os.listdir(d) if p.endswith(".cubin"))


def test_disk_cache_round_trip(tmp_path):
    first = _run(tmp_path)
    assert first["compiles"] == 1 and len(_files(tmp_path)) == 1
    second = _run(tmp_path)
    assert second["compiles"] == 0 and second["cache_hits"] == 1


@pytest.mark.parametrize("damage", ["flip", "truncate"])
def test_damaged_cache_file_is_recompiled(tmp_path, damage):
    _run(tmp_path)
    (name,) = _files(tmp_path)
    path = os.path.join(tmp_path, name)
    data = bytearray(open(path, "rb").read())
    good = bytes(data)
    if damage == "flip":
        data[len(data) // 2] ^= 0x5A  # inside the CUBIN, behind a valid header
    else:
        data = data[: len(data) - 100]
    open(path, "wb").write(bytes(data))
    again = _run(tmp_path)
    assert again["compiles"] == 1  # recompiled, not loaded
    assert open(path, "rb").read() == good  # and the file rewritten whole
    assert _run(tmp_path)["compiles"] == 0


def test_other_kernel_headers_do_not_share_cache_entries(tmp_path):
    # a copy of the library whose common header carries one extra line: the
    # generated source is the same, the headers it includes are not
    copy = tmp_path / "lib"
    shutil.copytree(os.path.join(ROOT, "elementwise_chain_jit_gb300"),
                    copy / "elementwise_chain_jit_gb300",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "include"), copy / "include")
    hdr = copy / "elementwise_chain_jit_gb300" / "csrc" / "kernels" / "common.cuh"
    hdr.write_text(hdr.read_text() + "// another build\n")
    subprocess.run([sys.executable, str(copy / "elementwise_chain_jit_gb300" / "buildlib.py")],
                   check=True, capture_output=True, timeout=600)
    cache = tmp_path / "cache"
    cache.mkdir()
    assert _run(cache)["compiles"] == 1
    assert _run(cache, root=str(copy))["compiles"] == 1  # not the other build's CUBIN
    assert len(_files(cache)) == 2
    assert _run(cache)["compiles"] == 0 and _run(cache, root=str(copy))["compiles"] == 0


def test_unwritable_cache_dir_is_ignored(tmp_path):
    blocker = tmp_path / "a_file"
    blocker.write_text("not a directory")
    stats = _run(blocker / "cache")  # a directory under a regular file cannot exist
    assert stats["compiles"] == 1


def test_forced_nvrtc_failure_reports_the_log(monkeypatch):
    monkeypatch.setenv("FUSE_NVRTC_OPTIONS", "--no-such-nvrtc-option")
    with pytest.raises(F.FuseError) as e:
        F.fuse_compile("relu;scale:0.625", (777,), F.F32)
    assert e.value.code == -6 and "NVRTC" in str(e.value)
    monkeypatch.delenv("FUSE_NVRTC_OPTIONS")
    c = F.fuse_compile("relu;scale:0.625", (777,), F.F32)  # the library is still usable
    assert c.n_in == 1
