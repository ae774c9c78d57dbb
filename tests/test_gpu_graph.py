"""GPU tests of fuse_graph_*: a sequence of library launches recorded with
stream capture and replayed as one graph.  Every replay's outputs are checked
against the oracle (the tolerances of the eager tests), and must also equal,
bit for bit, what the same launches produce when issued one by one."""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import tolerance as tol
import workloads
from gpu_util import to_host
from test_gpu_fixed import _rope_check
from test_gpu_rms_linear import _check as _rms_linear_check

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
    h_in1 = [to_host(t, d) for t, d in zip(in1, c1.in_dtypes)]
    h_in2 = to_host(in2, F.F16)
    hx, hr, hw = (to_host(t, F.BF16) for t in (x, r, w))
    y_want, h_want = oracle.rmsnorm_residual(hx, hr, hw, F.BF16, 1e-6)
    h_qkv = to_host(qkv, F.BF16)

    def check_against_oracle():
        for spec, dt, ins, shp, out, odt in ((spec1, dt1, h_in1, (n,), o1, c1.out_dtype),
                                             ("shuffle:4;relu;scale:0.5", F.F16, [h_in2], shape,
                                              o2, F.F16)):
            fails, counts, _ = oracle.chain_check(spec, dt, ins, shp, to_host(out, odt))
            assert fails == 0 and counts[3] == 0, (spec, counts)
        assert np.array_equal(to_host(ro, F.BF16), oracle.store(h_want, F.BF16))
        tol.assert_accepted(to_host(y, F.BF16), F.BF16, y_want, what="rmsnorm y")
        _rope_check(h_qkv, H, D, 5, F.BF16, *(to_host(t, F.BF16) for t in (q, k, v)))

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
        check_against_oracle()
        for a, b in zip(outs, want):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        for t in outs:
            t.zero_()
        torch.cuda.synchronize()
    g.release()


def test_graph_with_layernorm_detect_shuffle_and_tensor_core_kernels():
    """A captured sequence with the LayerNorm and detect kernels, a plain
    ChannelShuffle, and the tcgen05 RMSNorm -> Linear on both of its paths:
    folded weight (one cluster launch) and gamma per call, whose scratch copy
    of w is allocated and freed on the stream (memory nodes in the graph)."""
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    rows, hidden = 40, 2048
    x = workloads.device_normal((rows, hidden), 0, 1, 71, F.BF16)
    r = workloads.device_normal((rows, hidden), 0, 1, 72, F.BF16)
    g = workloads.device_normal((hidden,), 1, 0.1, 73, F.BF16)
    b = workloads.device_normal((hidden,), 0, 0.1, 74, F.BF16)
    ly, lro = torch.empty_like(x), torch.empty_like(x)
    hw, strides, na, no = [(8, 8), (4, 4)], [8.0, 16.0], 3, 85
    anchors = workloads.detect_anchors(strides, na)
    feats = [workloads.device_normal((1, na * no, h, w_), 0, 2, 75 + i, F.F16)
             for i, (h, w_) in enumerate(hw)]
    dout = torch.empty(sum(na * h * w_ for h, w_ in hw) * no, dtype=torch.float32, device=dev)
    dec = F.DetectDecoder(hw, strides, anchors, na, no, F.F16)
    sx = workloads.device_uniform(2 * 16 * 8 * 8, -2, 2, 77, F.F16)
    so = torch.empty_like(sx)
    M, N, K = 300, 264, 136
    xm = workloads.device_normal((M, K), 0, 1, 78, F.BF16)
    gm = workloads.device_normal((K,), 1, 0.1, 79, F.BF16)
    wm = workloads.device_normal((N, K), 0, K ** -0.5, 80, F.BF16)
    bm = workloads.device_normal((N,), 0, 0.5, 81, F.BF16)
    wf = torch.empty_like(wm)
    F.rmsnorm_linear_fold(wm, gm, wf, F.BF16)
    o_fold = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    o_gamma = torch.empty_like(o_fold)

    def sequence():
        F.layernorm_residual(x, r, g, b, ly, lro, 1e-5, F.BF16, stream=s)
        dec(feats, dout, stream=s)
        F.channel_shuffle(sx, so, 4, F.F16, shape=(2, 16, 8, 8), stream=s)
        F.rmsnorm_linear(xm, None, wf, bm, o_fold, 1e-6, 0.5, F.BF16, stream=s)
        F.rmsnorm_linear(xm, gm, wm, bm, o_gamma, 1e-6, 0.5, F.BF16, stream=s)

    outs = [ly, lro, dout, so, o_fold, o_gamma]
    hx, hr, hg, hb = (to_host(t, F.BF16) for t in (x, r, g, b))
    ln_want, ln_h, ln_mag = oracle.layernorm_residual(hx, hr, hg, hb, F.BF16, 1e-5)
    d_want, d_mag = oracle.detect_decode([to_host(f, F.F16).reshape(1, na * no, h, w_)
                                          for f, (h, w_) in zip(feats, hw)],
                                         F.F16, strides, anchors, na, no)
    s_want = oracle.channel_shuffle(to_host(sx, F.F16).reshape(2, 16, 8, 8), 4)
    hxm, hgm, hwm, hbm = (to_host(t, F.BF16) for t in (xm, gm, wm, bm))
    m_want, m_mag = oracle.rmsnorm_linear(hxm, hgm, hwm, hbm, F.BF16, 1e-6, 0.5)

    def check_against_oracle():
        assert np.array_equal(to_host(lro, F.BF16), oracle.store(ln_h, F.BF16))
        tol.assert_accepted(to_host(ly, F.BF16), F.BF16, ln_want, ln_mag, what="layernorm")
        tol.assert_accepted(to_host(dout, F.F32), F.F32, d_want.reshape(-1), d_mag.reshape(-1),
                            what="detect")
        assert np.array_equal(to_host(so, F.F16), s_want.reshape(-1))
        for o in (o_fold, o_gamma):
            _rms_linear_check(to_host(o, F.BF16), F.BF16, hxm, m_want, m_mag, 0.5, K)

    with torch.cuda.stream(s):
        sequence()
    s.synchronize()
    assert F.fuse_device_error() == 0
    want = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    torch.cuda.synchronize()
    F.fuse_graph_begin(s)
    sequence()
    gr = F.fuse_graph_end(s)
    assert gr.nodes >= 6  # six kernels, plus the gamma path's memory nodes
    for _ in range(3):
        gr.launch(s)
        s.synchronize()
        check_against_oracle()
        for a, w_ in zip(outs, want):
            assert torch.equal(a.view(torch.uint8), w_.view(torch.uint8))
        for t in outs:
            t.zero_()
        torch.cuda.synchronize()
    assert F.fuse_device_error() == 0
    gr.release()
