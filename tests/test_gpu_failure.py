"""The failure path of the kernels' bounded waits, on the GPU: a wait on an
mbarrier that nothing arrives at (the library's bounded wait, in the
fuse_selftest_bounded_wait kernel) gives up, records code 1 in the device
error word, and the context stays usable.  No fault, trap or hang is caused.
"""
import time

import pytest
import torch

import elementwise_chain_jit_gb300 as F

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("spins", [1, 1 << 12, 1 << 16])
def test_bounded_wait_gives_up_and_reports(spins):
    F.fuse_device_error()  # clear
    F.fuse_selftest_bounded_wait(spins)
    torch.cuda.synchronize()
    assert F.fuse_device_error() == 1
    assert F.fuse_device_error() == 0  # reading clears the word
    # the context is still usable: a chain runs and is bit-exact
    g = torch.Generator(device="cuda").manual_seed(5)
    a = torch.rand(4099, device="cuda", generator=g) * 2 - 1
    b = torch.rand(4099, device="cuda", generator=g) * 2 - 1
    out = torch.empty_like(a)
    F.fuse_launch(F.fuse_compile("add;relu;scale:0.5", a.shape, F.F32), [a, b], out)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.relu(a + b) * 0.5)
    assert F.fuse_device_error() == 0


def test_the_kernels_bound_ends_within_seconds():
    # 2^18 tries: the bound of every wait inside the tcgen05 kernels
    F.fuse_device_error()
    t0 = time.perf_counter()
    F.fuse_selftest_bounded_wait(1 << 18)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert F.fuse_device_error() == 1
    print(f"bounded wait of 2^18 tries gave up after {took:.3f} s")
    assert took < 10
