"""Dynamic shapes on the fixed entry points: one compile serves every token
count of rope_qkv_split and every batch size of channel_shuffle ("DeepJIT",
section 7.2: quantise dynamic shapes so that the hot path never compiles;
section 6.2: keep compiling off the request path).  Every call is checked
against the oracle, and the library's compile counter must move by exactly
one over all of them."""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads
from gpu_util import to_dev, to_host
from test_gpu_fixed import _rope_check

pytestmark = pytest.mark.gpu


def test_rope_token_counts_1_to_257_compile_once():
    heads, hd, dt = 3, 72, F.F16  # a shape no other test uses
    # any first RoPE call compiles the table builder once per process; make
    # it on another head count, so that only the kernel under test is new
    warm = torch.zeros(3 * 5 * hd, dtype=torch.float16, device="cuda")
    outs = [torch.empty(5 * hd, dtype=torch.float16, device="cuda") for _ in range(3)]
    F.rope_qkv_split(warm, *outs, 5, hd, 0, 10000.0, dt, tokens=1)
    torch.cuda.synchronize()
    before = F.fuse_stats()["compiles"]
    for tokens in range(1, 258):
        pos0 = (tokens * 7919) % 30000
        qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, 5000 + tokens, dt)
        q, k, v = (torch.empty(heads * tokens * hd, dtype=torch.float16, device="cuda")
                   for _ in range(3))
        F.rope_qkv_split(to_dev(qkv.reshape(-1), dt), q, k, v, heads, hd, pos0, 10000.0, dt,
                         tokens=tokens)
        torch.cuda.synchronize()
        _rope_check(qkv, heads, hd, pos0, dt, *(to_host(t, dt) for t in (q, k, v)))
    assert F.fuse_stats()["compiles"] - before == 1


@pytest.mark.parametrize("dt", [F.F16, F.F32])
def test_channel_shuffle_batches_1_to_32_compile_once(dt):
    c, h, w, g = 24, 5, 8, 3  # a shape no other test uses (H*W a multiple of 8)
    if dt == F.F32:
        w = 7  # odd plane: the scalar kernel of the same bucket module
    before = F.fuse_stats()["compiles"]
    for n in range(1, 33):
        x = workloads.uniform(n * c * h * w, -2, 2, 6000 + n, dt).reshape(n, c, h, w)
        out = torch.empty(n * c * h * w, dtype=torch.float32 if dt == F.F32 else torch.float16,
                          device="cuda")
        F.channel_shuffle(to_dev(x.reshape(-1), dt), out, g, dt, shape=(n, c, h, w))
        torch.cuda.synchronize()
        want = oracle.channel_shuffle(x, g)
        assert np.array_equal(to_host(out, dt).reshape(n, c, h, w).view(np.uint8),
                              want.view(np.uint8)), n
    assert F.fuse_stats()["compiles"] - before == 1
