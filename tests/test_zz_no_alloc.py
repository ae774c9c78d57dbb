"""rope_qkv_split_noalloc: the allocation-free variant of QKV split + RoPE.

Callers that cannot let a library allocate device memory -- a server whose
device memory is all owned by its own caching allocator, code running inside
a CUDA-graph stream capture, loops that forbid allocation after start-up --
call this entry point instead of rope_qkv_split.  Its cos/sin rows live in a
fixed 4 MB array inside the library's module; every call shares it.

The tests call it through the C ABI and check every result against the
oracle: v bit for bit, q and k within the RoPE tolerance (tests/tolerance.py:
8e-3 relative to the magnitude of the rotation's two terms for bf16, 2 ulp
for fp16, 1e-6 for fp32).
  * After one set-up call (bf16), calls of all three dtypes are recorded into
    a CUDA graph with stream capture (thread-local mode: an allocation or a
    synchronising call of this thread inside the capture breaks it) and
    replayed twice; the same calls made eagerly change neither PyTorch's
    allocated memory nor the device's free memory.
  * Two calls in a row for each dtype, on different inputs, positions and
    token counts, so the second call runs over rows the first one left
    behind (16-byte vector kernel), and the element-wise kernel on an odd
    half row and on tensors off the 16-byte boundary.
  * A call larger than the fixed array is refused with FUSE_E_SHAPE.
The file is named to be collected last; it needs nothing from earlier tests
and passes alone in a fresh process.
"""
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import workloads
from gpu_util import Guarded, misaligned_copy, to_dev, to_host
from test_gpu_fixed import _rope_check, _table_check

pytestmark = pytest.mark.gpu

DTS = [F.F32, F.F16, F.BF16]
TORCH_DT = {F.F32: torch.float32, F.F16: torch.float16, F.BF16: torch.bfloat16}


def _case(tokens, heads, hd, dt, seed):
    qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, seed, dt)
    outs = [torch.full((heads * tokens * hd,), float("nan"), dtype=TORCH_DT[dt], device="cuda")
            for _ in range(3)]
    return qkv, to_dev(qkv.reshape(-1), dt), outs


def test_noalloc_calls_in_a_captured_graph_allocate_nothing():
    heads, hd = 4, 128
    # set-up call (first in this context, any dtype)
    qkv0, qd0, o0 = _case(64, heads, hd, F.BF16, 880)
    F.rope_qkv_split_noalloc(qd0, *o0, heads, hd, 100, 10000.0, F.BF16, tokens=64)
    torch.cuda.synchronize()
    _rope_check(qkv0, heads, hd, 100, F.BF16, *(to_host(t, F.BF16) for t in o0))

    cases = [(dt, 40 + 24 * i, 1000 * (i + 1)) + _case(40 + 24 * i, heads, hd, dt, 890 + i)
             for i, dt in enumerate(DTS)]
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    for dt, tokens, pos0, _, qd, outs in cases:  # eager, every dtype
        F.rope_qkv_split_noalloc(qd, *outs, heads, hd, pos0, 10000.0, dt, tokens=tokens)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    for dt, tokens, pos0, qkv, _, outs in cases:
        _rope_check(qkv, heads, hd, pos0, dt, *(to_host(t, dt) for t in outs))
        for t in outs:
            t.fill_(float("nan"))

    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    F.fuse_graph_begin(s)
    for dt, tokens, pos0, _, qd, outs in cases:
        F.rope_qkv_split_noalloc(qd, *outs, heads, hd, pos0, 10000.0, dt, tokens=tokens, stream=s)
    g = F.fuse_graph_end(s)
    assert g.nodes == 2 * len(cases)  # the rows build and the rotation, per call
    for _ in range(2):
        g.launch(s)
        s.synchronize()
        for dt, tokens, pos0, qkv, _, outs in cases:
            _rope_check(qkv, heads, hd, pos0, dt, *(to_host(t, dt) for t in outs))
            for t in outs:
                t.fill_(float("nan"))
        torch.cuda.synchronize()
    g.release()


@pytest.mark.parametrize("dt", DTS)
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(dt):
    heads, hd = 8, 128
    for call, (tokens, pos0) in enumerate([(1024, 31000), (300, 7)]):
        qkv, qd, outs = _case(tokens, heads, hd, dt, 900 + call + 10 * dt)
        F.rope_qkv_split_noalloc(qd, *outs, heads, hd, pos0, 10000.0, dt, tokens=tokens)
        torch.cuda.synchronize()
        _rope_check(qkv, heads, hd, pos0, dt, *(to_host(t, dt) for t in outs))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("tokens,heads,hd,offset", [(33, 3, 6, 0), (17, 2, 128, 1)])
def test_noalloc_element_wise_path(dt, tokens, heads, hd, offset):
    """Half a row that is not a whole number of 16-byte vectors, or tensors
    off the 16-byte boundary: the element-wise kernel, against the oracle."""
    qkv, qd, _ = _case(tokens, heads, hd, dt, 950 + hd + offset)
    if offset:
        qd = misaligned_copy(qd, offset)
    outs = [Guarded(heads * tokens * hd, dt, offset_elems=offset) for _ in range(3)]
    F.rope_qkv_split_noalloc(qd, *(o.t for o in outs), heads, hd, 77, 10000.0, dt, tokens=tokens)
    torch.cuda.synchronize()
    assert all(o.canary_ok() for o in outs)
    _rope_check(qkv, heads, hd, 77, dt, *(to_host(o.t, dt) for o in outs))


@pytest.mark.parametrize("pos0", [0, 1000, (1 << 22) - 2048])
def test_noalloc_rows_are_correctly_rounded(pos0):
    """The cos/sin rows it builds per call (reduced argument, Taylor series in
    binary64) are the fp32 values nearest the exact ones, up to the largest
    positions."""
    _table_check(F.rope_qkv_split_noalloc, 2048, pos0)


def test_noalloc_refuses_calls_beyond_its_fixed_array():
    with pytest.raises(F.FuseError) as e:
        F.rope_qkv_split_noalloc(256, 256, 256, 256, 4, 128, 0, 10000.0, F.BF16,
                                 tokens=(1 << 20) // 128 + 1, stream=0)
    assert e.value.code == -2 and "fixed table" in str(e.value)
