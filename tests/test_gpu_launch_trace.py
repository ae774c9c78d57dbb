"""The launch counts the bench reports, checked against a timeline trace
(CUPTI records through torch.profiler): each fused workload is exactly one
device activity, and each unfused sequence launches the number of kernels
the bench declares for it."""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu

SMALL = (r"add_relu_scale|detect_decode|shuffle_chain_L4$|flat_chain_L2_|rmsnorm_residual|rope_qkv"
         r"|channel_shuffle")


@pytest.fixture(scope="module")
def items():
    dev = torch.device("cuda", 0)
    its = bench.build_items(dev, with_unfused=True, only=SMALL, flat_elems=(1 << 20) + 7)
    its.append(bench._ln_item(dev, with_unfused=True))
    its.append(bench._rms_linear_item(dev, with_unfused=True, M=256))
    bench.device_ops(lambda: None)  # the first session of a process can miss records
    return its


def test_fused_is_one_launch_and_unfused_counts_match(items):
    assert len(items) == 9
    for it in items:
        it.fused()
        ops = bench.device_ops(it.fused)
        assert len(ops) == 1, (it.name, ops)
        it.unfused()
        ops = bench.device_ops(it.unfused)
        assert len(ops) == it.n_unfused, (it.name, len(ops), [o[2][:40] for o in ops])
