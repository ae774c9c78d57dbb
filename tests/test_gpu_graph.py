"""GPU tests of fuse_graph_*: a sequence of library launches recorded with
stream capture and replayed as one graph must produce exactly what the same
launches produce when issued one by one."""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import workloads

pytestmark = pytest.mark.gpu


def test_graph_replays_a_mixed_sequence_bit_exactly():
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    n = 100_003
    spec1, dt1 = workloads.random_chain(8, 21)
    c1 = F.fuse_compile(spec1, (n,), dt1)
    in1 = [workloads.device_uniform(n, -2, 2, 50 + j, d) for j, d in enumerate(c1.in_dtypes)]
    o1 = torch.empty(n, dtype={0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[c1.out_dtype],
                     device=dev)
    shape = (4, 16, 8, 8)
    c2 = F.fuse_compile("shuffle:4;relu;scale:0.5", shape, F.F16)
    in2 = workloads.device_uniform(int(np.prod(shape)), -2, 2, 60, F.F16)
    o2 = torch.empty_like(in2)
    rows, hidden = 33, 4096
    x = workloads.device_normal((rows, hidden), 0, 1, 61, F.BF16)
    r = workloads.device_normal((rows, hidden), 0, 1, 62, F.BF16)
    w = workloads.device_normal((hidden,), 1, 0.1, 63, F.BF16)
    y, ro = torch.empty_like(x), torch.empty_like(x)
    T, H, D = 17, 4, 128
    qkv = workloads.device_normal((T, 3 * H * D), 0, 1, 64, F.BF16)
    q, k, v = (torch.empty(H * T * D, dtype=torch.bfloat16, device=dev) for _ in range(3))

    def sequence():
        F.fuse_launch(c1, in1, o1, stream=s)
        F.fuse_launch(c2, [in2], o2, stream=s)
        F.rmsnorm_residual(x, r, w, y, ro, 1e-6, F.BF16, stream=s)
        F.rope_qkv_split(qkv, q, k, v, H, D, 5, 10000.0, F.BF16, stream=s)

    outs = [o1, o2, y, ro, q, k, v]
    with torch.cuda.stream(s):
        sequence()  # first use: compiles, loads modules, builds the RoPE table
    s.synchronize()
    want = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    torch.cuda.synchronize()
    F.fuse_graph_begin(s)
    sequence()
    g = F.fuse_graph_end(s)
    assert g.nodes == 4
    s.synchronize()
    assert all(not torch.equal(a, b) for a, b in zip(outs, want))  # still zeroed
    for _ in range(2):
        g.launch(s)
        s.synchronize()
        for a, b in zip(outs, want):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        for t in outs:
            t.zero_()
        torch.cuda.synchronize()
    g.release()
