"""Seeded random shapes through the fixed entry points, against the oracle:
residual + RMSNorm and LayerNorm (any row length, row count, dtype, alignment),
QKV split + RoPE (even head dims, head counts, token counts, start positions)
and the detection decode (one to four scales of any size, anchors and outputs
per cell).  The helpers are the ones of test_gpu_fixed, tolerances included."""
import numpy as np
import pytest
import torch

import elementwise_chain_jit_gb300 as F
import workloads
from gpu_util import Guarded, misaligned_copy, to_dev, to_host
from test_gpu_fixed import _detect_case, _ln_case, _rms_case, _rope_check

pytestmark = pytest.mark.gpu

DTS = (F.BF16, F.F16, F.F32)


@pytest.mark.parametrize("block", range(2))
def test_norms_random_shapes(block):
    rng = np.random.default_rng(800 + block)
    for i in range(10):
        rows = int(rng.integers(1, 300))
        hidden = int(rng.choice([int(rng.integers(1, 9000)), 8 * int(rng.integers(1, 1100))]))
        dt = DTS[int(rng.integers(0, 3))]
        offset = int(rng.random() < 0.25)
        seed = 900 + 20 * block + i
        _rms_case(rows, hidden, dt, seed, offset=offset)
        _ln_case(rows, hidden, dt, seed, flags=int(rng.integers(0, 8)), offset=offset)


@pytest.mark.parametrize("block", range(2))
def test_rope_random_shapes(block):
    rng = np.random.default_rng(820 + block)
    for i in range(10):
        tokens = int(rng.integers(1, 200))
        heads = int(rng.integers(1, 17))
        hd = 2 * int(rng.integers(1, 129))
        pos0 = int(rng.integers(0, 40000))
        dt = DTS[int(rng.integers(0, 3))]
        offset = int(rng.random() < 0.25)
        qkv = workloads.normal((tokens, 3 * heads * hd), 0, 1, 950 + 20 * block + i, dt)
        qd = to_dev(qkv.reshape(-1), dt)
        if offset:
            qd = misaligned_copy(qd, 1)
        outs = [Guarded(heads * tokens * hd, dt, offset_elems=offset) for _ in range(3)]
        F.rope_qkv_split(qd, outs[0].t, outs[1].t, outs[2].t, heads, hd, pos0, 10000.0, dt,
                         tokens=tokens)
        torch.cuda.synchronize()
        assert all(o.canary_ok() for o in outs)
        _rope_check(qkv, heads, hd, pos0, dt, *(to_host(o.t, dt) for o in outs))


@pytest.mark.parametrize("block", range(2))
def test_detect_random_shapes(block):
    rng = np.random.default_rng(840 + block)
    for i in range(8):
        ns = int(rng.integers(1, 5))
        hw = [(int(rng.integers(1, 41)), int(rng.integers(1, 41))) for _ in range(ns)]
        na = int(rng.integers(1, 5))
        no = int(rng.integers(5, 100))
        dt = DTS[int(rng.integers(0, 3))]
        offset = int(rng.random() < 0.25)
        _detect_case(hw, dt, 980 + 20 * block + i, offset=offset, na=na, no=no)
