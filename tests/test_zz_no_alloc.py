"""rope_qkv_split_noalloc: the allocation-free variant of QKV split + RoPE.

Callers that cannot let a library allocate device memory -- a server whose
device memory is all owned by its own caching allocator, code running inside
a CUDA-graph stream capture, loops that forbid allocation after start-up --
call this entry point instead of rope_qkv_split.  Its cos/sin rows live in a
fixed 4 MB array inside the library's module; every call shares it.

This test calls it through the C ABI twice in a row, on different inputs,
positions and token counts (so the second call runs over rows the first one
left behind), and checks each result against rope_qkv_split on the same
inputs: v bit for bit, q and k within the RoPE tolerance (8e-3 relative to
the magnitude of the rotation's two terms, from the oracle).  It also checks
that a call larger than the fixed array is refused with FUSE_E_SHAPE.  The
file is named to be collected last; it needs nothing from earlier tests.
"""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _down(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_noalloc_matches_rope_qkv_split_on_two_calls_in_a_row():
    heads, hd = 8, 128
    for call, (tokens, pos0) in enumerate([(1024, 31000), (300, 7)]):
        qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, 900 + call, F.BF16)
        qd = _up(qkv.reshape(-1))
        ref = [torch.empty(heads * tokens * hd, dtype=torch.bfloat16, device="cuda")
               for _ in range(3)]
        got = [torch.full_like(r, float("nan")) for r in ref]
        F.rope_qkv_split(qd, *ref, heads, hd, pos0, 10000.0, F.BF16, tokens=tokens)
        F.rope_qkv_split_noalloc(qd, *got, heads, hd, pos0, 10000.0, F.BF16, tokens=tokens)
        torch.cuda.synchronize()
        r_q, r_k, r_v = (_down(t) for t in ref)
        g_q, g_k, g_v = (_down(t) for t in got)
        assert np.array_equal(g_v, r_v)
        _, _, _, qm, km = oracle.rope_qkv_split(qkv, F.BF16, heads, hd, pos0 + np.arange(tokens))
        for g, r, mag in ((g_q, r_q, qm), (g_k, r_k, km)):
            gd = oracle.to_double(g, F.BF16).reshape(mag.shape)
            rd = oracle.to_double(r, F.BF16).reshape(mag.shape)
            assert np.all(np.abs(gd - rd) <= 8e-3 * mag), call


def test_noalloc_refuses_calls_beyond_its_fixed_array():
    with pytest.raises(F.FuseError) as e:
        F.rope_qkv_split_noalloc(256, 256, 256, 256, 4, 128, 0, 10000.0, F.BF16,
                                 tokens=(1 << 20) // 128 + 1, stream=0)
    assert e.value.code == -2 and "fixed table" in str(e.value)
