"""Several host threads using the library at once, each on its own stream.

Each thread compiles its chains (sources shared between threads compile once),
launches them repeatedly on its own CUDA stream and checks the result against
the oracle; a warm-up list compiled beforehand leaves nothing to compile.
"""
import concurrent.futures as cf

import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads
from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def _job(k):
    spec, dt = workloads.random_chain(4 + 4 * (k % 4), 40 + k % 4)
    n = 10_007 + 96 * k
    inputs, _ = workloads.chain_inputs(spec, dt, n, 50 + k)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        c = F.fuse_compile(spec, (n,), dt)
        dev = [to_dev(a, d) for a, d in zip(inputs, c.in_dtypes)]
        out = torch.empty(n, dtype={0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[c.out_dtype],
                          device="cuda")
        for _ in range(25):
            F.fuse_launch(c, dev, out)
        stream.synchronize()
        got = to_host(out, c.out_dtype)
    fails, counts, _ = oracle.chain_check(spec, dt, inputs, (n,), got)
    return fails, counts[3]


def test_threads_each_on_their_own_stream():
    with cf.ThreadPoolExecutor(8) as pool:
        results = list(pool.map(_job, range(16)))
    assert all(f == 0 for f, _ in results), results
    assert all(u == 0 for _, u in results), results  # none unpinned


def test_warmed_up_chains_launch_without_compiling():
    entries = [(f"add;sigmoid;scale:{k + 2}.5", (4096,), F.F32) for k in range(4)]
    F.fuse_warmup(entries, threads=4)
    before = F.fuse_stats()["compiles"]
    for spec, shape, dt in entries:
        a = workloads.uniform(shape[0], -2, 2, 7, F.F32)
        b = workloads.uniform(shape[0], -2, 2, 8, F.F32)
        c = F.fuse_compile(spec, shape, dt)
        out = torch.empty(shape[0], dtype=torch.float32, device="cuda")
        F.fuse_launch(c, [to_dev(a, F.F32), to_dev(b, F.F32)], out)
        torch.cuda.synchronize()
        fails, counts, _ = oracle.chain_check(spec, dt, [a, b], shape, to_host(out, F.F32))
        assert fails == 0 and counts[3] == 0, counts
    assert F.fuse_stats()["compiles"] == before
