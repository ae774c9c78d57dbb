"""Producer -> consumer launches back to back on one stream, with no host
synchronisation between them.

Every library kernel is launched with programmatic dependent launch: its CTAs
may start while the previous kernel drains, and before waiting for it they
prefetch their first chunk or row into L2.  These tests check that a consumer
still reads what its producer wrote, every time: each round overwrites the
producer's output with new values, and each consumer result is checked
against the oracle on a sample of its elements (the ends, the first chunks,
which are the prefetched ones, and random positions).
"""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import oracle
import tolerance as tol
import workloads
from gpu_util import to_host

pytestmark = pytest.mark.gpu


def _sample(n, seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(min(n, 1 << 16)), np.arange(n - 4096, n),
                                     g.integers(0, n, 50_000)]))


def test_chain_reads_what_the_previous_chain_wrote():
    n = (1 << 24) + 7
    prod = F.fuse_compile("add;relu", (n,), F.F32)
    cons = F.fuse_compile("mul;sigmoid;cast:f16", (n,), F.F32)
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    c = workloads.device_uniform(n, -2, 2, 7, F.F32)
    rounds = []
    for r in range(4):
        a = workloads.device_uniform(n, -2, 2, 100 + r, F.F32)
        b = workloads.device_uniform(n, -2, 2, 200 + r, F.F32)
        z = torch.empty(n, dtype=torch.float16, device="cuda")
        F.fuse_launch(prod, [a, b], y)   # y is overwritten every round
        F.fuse_launch(cons, [y, c], z)   # and read at once, no sync between
        rounds.append((a, b, z))
    torch.cuda.synchronize()
    idx = _sample(n, 1)
    it = torch.from_numpy(idx).cuda()
    hc = to_host(c[it], F.F32)
    for a, b, z in rounds:
        ha, hb = to_host(a[it], F.F32), to_host(b[it], F.F32)
        # the pair as one chain: relu(a + b) * c -> sigmoid -> f16
        fails, counts, _ = oracle.chain_check("add;relu;mul;sigmoid;cast:f16", F.F32, [ha, hb, hc],
                                              (len(idx),), to_host(z[it], F.F16))
        assert fails == 0 and counts[3] == 0, counts


def test_fixed_ops_read_what_a_chain_wrote():
    rows, hidden = 8192, 4096
    T, H, D = 4096, 32, 128
    mk = F.fuse_compile("scale:0.5", (rows * hidden,), F.BF16)
    mq = F.fuse_compile("scale:0.5", (T * 3 * H * D,), F.BF16)
    x = torch.empty(rows * hidden, dtype=torch.bfloat16, device="cuda")
    qkv = torch.empty(T * 3 * H * D, dtype=torch.bfloat16, device="cuda")
    r = workloads.device_normal((rows, hidden), 0, 1, 11, F.BF16)
    w = workloads.device_normal((hidden,), 1, 0.1, 12, F.BF16)
    outs = []
    for k in range(3):
        xs = workloads.device_normal((rows * hidden,), 0, 1, 20 + k, F.BF16)
        qs = workloads.device_normal((T * 3 * H * D,), 0, 1, 30 + k, F.BF16)
        y, ro = torch.empty_like(x), torch.empty_like(x)
        q, kk, v = (torch.empty(H * T * D, dtype=torch.bfloat16, device="cuda") for _ in range(3))
        F.fuse_launch(mk, [xs], x)        # x = xs / 2, then RMSNorm reads x at once
        F.rmsnorm_residual(x, r, w, y, ro, 1e-6, F.BF16, rows=rows, hidden=hidden)
        F.fuse_launch(mq, [qs], qkv)      # qkv = qs / 2, then RoPE reads it at once
        F.rope_qkv_split(qkv, q, kk, v, H, D, 0, 10000.0, F.BF16, tokens=T)
        outs.append((xs, qs, y, ro, q, kk, v))
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([[0, 1, 2, rows - 1], np.random.default_rng(2).integers(0, rows, 29)]))
    tsel = np.unique(np.concatenate([[0, 1, T - 1], np.random.default_rng(3).integers(0, T, 29)]))
    st, tt = torch.from_numpy(sel).cuda(), torch.from_numpy(tsel).cuda()
    hr, hw = to_host(r[st], F.BF16), to_host(w, F.BF16)
    for xs, qs, y, ro, q, kk, v in outs:
        hx = oracle.store(oracle.to_double(to_host(xs.view(rows, hidden)[st], F.BF16), F.BF16) * 0.5,
                          F.BF16)
        yw, hh = oracle.rmsnorm_residual(hx, hr, hw, F.BF16, 1e-6)
        assert np.array_equal(to_host(ro.view(rows, hidden)[st], F.BF16), oracle.store(hh, F.BF16))
        tol.assert_accepted(to_host(y.view(rows, hidden)[st], F.BF16), F.BF16, yw, what="rmsnorm")
        hq = oracle.store(oracle.to_double(to_host(qs.view(T, 3 * H * D)[tt], F.BF16), F.BF16) * 0.5,
                          F.BF16)
        qw, kw, vw, qm, km = oracle.rope_qkv_split(hq, F.BF16, H, D, tsel)
        sub = lambda t: to_host(t.view(H, T, D)[:, tt].contiguous(), F.BF16)  # noqa: E731
        tol.assert_accepted(sub(q), F.BF16, qw, qm, what="rope q")
        tol.assert_accepted(sub(kk), F.BF16, kw, km, what="rope k")
        assert np.array_equal(sub(v).reshape(vw.shape), oracle.store(vw, F.BF16))
