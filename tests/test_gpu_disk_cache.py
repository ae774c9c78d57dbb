"""The compiled-code disk cache on the GPU ("DeepJIT", section 6.2: keep
compiled code on disk so that a restarted process does not compile again).

Process A compiles a chain and an RMSNorm kernel with FUSE_CACHE_DIR set (and
runs them).  Process B, a fresh process on the same directory, must take both
kernels from the disk (no NVRTC compile), launch them, and produce outputs
that pass the oracle: the chain through the chain check (bit-exact or within
the error bound), RMSNorm at the stated tolerances and its updated residual
bit for bit."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SPEC = "add;exp;scale:0.8125;mul;sigmoid;cast:f16"  # a chain no other test compiles

SCRIPT = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import torch
import elementwise_chain_jit_gb300 as F
import oracle, workloads
import tolerance as tol
from gpu_util import to_dev, to_host
n = 70001
spec, dt = {spec!r}, F.F32
ins, dts = workloads.chain_inputs(spec, dt, n, 4242)
c = F.fuse_compile(spec, (n,), dt)
out = torch.empty(n, dtype=torch.float16, device="cuda")
F.fuse_launch(c, [to_dev(a, d) for a, d in zip(ins, dts)], out)
rows, hidden = 37, 2304
x = workloads.normal((rows, hidden), 0, 1, 4243, F.BF16)
r = workloads.normal((rows, hidden), 0, 1, 4244, F.BF16)
w = workloads.normal(hidden, 1, 0.1, 4245, F.BF16)
y = torch.empty(rows * hidden, dtype=torch.bfloat16, device="cuda")
ro = torch.empty_like(y)
F.rmsnorm_residual(to_dev(x.reshape(-1), F.BF16), to_dev(r.reshape(-1), F.BF16),
                   to_dev(w, F.BF16), y, ro, 1e-6, F.BF16, rows=rows, hidden=hidden)
torch.cuda.synchronize()
fails, counts, _ = oracle.chain_check(spec, dt, ins, (n,), to_host(out, F.F16))
yw, hw = oracle.rmsnorm_residual(x, r, w, F.BF16, 1e-6)
rms_ok = bool(tol.accepted(to_host(y, F.BF16), F.BF16, yw.reshape(-1)).all())
res_ok = bool(np.array_equal(to_host(ro, F.BF16), oracle.store(hw, F.BF16).reshape(-1)))
print(json.dumps(dict(F.fuse_stats(), fails=int(fails), unpinned=int(counts[3]), rms_ok=rms_ok,
                      res_ok=res_ok)))
"""


def _run(cache_dir):
    env = dict(os.environ, FUSE_CACHE_DIR=str(cache_dir))
    env.pop("FUSE_NVRTC_OPTIONS", None)
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"), spec=SPEC)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-4000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_a_restarted_process_runs_kernels_from_the_disk_cache(tmp_path):
    a = _run(tmp_path)
    assert a["compiles"] == 2, a  # the chain and the RMSNorm kernel
    assert len([p for p in os.listdir(tmp_path) if p.endswith(".cubin")]) == 2
    b = _run(tmp_path)
    assert b["compiles"] == 0 and b["cache_hits"] >= 2, b
    for s in (a, b):
        assert s["fails"] == 0 and s["unpinned"] == 0 and s["rms_ok"] and s["res_ok"], s
