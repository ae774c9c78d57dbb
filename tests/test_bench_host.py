"""Host-side logic of bench.py (no GPU): the launch-cost model against the
page's worked numbers, and the CPU-oracle sample."""
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "launch_model.txt")


def test_launch_model_matches_page_numbers():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    k, tu, tf, L_page, T_page = rows[0]
    L, T = bench.launch_overhead(float(tu), float(tf), int(k))
    assert round(L, 3) == float(L_page)
    assert round(T, 2) == float(T_page)
    assert abs(int(k) * L + T - float(tu)) < 1e-12


def test_cpu_sample_is_bounded_and_positive():
    b, t, desc = bench.cpu_sample(4096)
    assert b > 0 and t > 0 and "rope" in desc


def test_reference_arm_prints_one_json_line(capsys):
    class A:
        gpus, steps, warmup = 1, 1, 0
    import json
    bench.run_reference(A())
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_mufu_operations_of_a_chain():
    # exp: one ex2; sigmoid: one ex2 and one rcp; the prologue, scale
    # constants, the fast forms' names and the other ops add nothing
    assert bench.mufu_ops_per_element("shuffle:4;exp") == (1, 0)
    assert bench.mufu_ops_per_element("relu;sigmoid") == (1, 1)
    assert bench.mufu_ops_per_element("exp:fast;sigmoid:fast;relu;mul") == (2, 1)
    assert bench.mufu_ops_per_element("cast:f32;scale:0.5;add;mul") == (0, 0)


def test_mufu_floor_adds_the_two_instructions_at_their_rates():
    rates = bench.nominal_mufu_rates(sms=152, mhz=2000.0)
    assert rates["ex2_per_s"] == 32 * 152 * 2e9 and rates["rcp_per_s"] == 16 * 152 * 2e9
    # 8 ex2 and 4 rcp per element, 2^20 elements: one SM-clock of unit time
    # per 2 elements on each SM
    us = bench.mufu_floor_us((8 << 20, 4 << 20), rates)
    assert us == pytest.approx((1 << 20) * 0.5 / (152 * 2e9) * 1e6)


def test_cpu_all_cores_sample_uses_every_core():
    b, t, threads, desc = bench.cpu_sample_all_cores(4096)
    assert b > 0 and t > 0 and threads == (os.cpu_count() or 1) and "slices" in desc


def test_link_bound_takes_the_slower_direction():
    step, h2d, d2h = 29.0e9, 22.7e9, 6.3e9
    # fast both ways: the inputs bind (22.7 GB at 210 GB/s)
    fast = bench.link_bound(step, 1, h2d, d2h, {"h2d": 210.0, "d2h": 193.0, "both": 340.0})
    assert fast == pytest.approx(step / (h2d / 210e9) / 1e9)
    # slow device-to-host: still the inputs (6.3 GB at 67 GB/s is 94 ms < 108 ms)
    slow = bench.link_bound(step, 1, h2d, d2h, {"h2d": 210.0, "d2h": 67.0, "both": 122.0})
    assert slow == pytest.approx(fast)
    # slower still: the outputs bind
    slower = bench.link_bound(step, 1, h2d, d2h, {"h2d": 210.0, "d2h": 20.0, "both": 100.0})
    assert slower == pytest.approx(step / (d2h / 20e9) / 1e9)
    # two ranks move twice the bytes in the same time
    assert bench.link_bound(step, 2, h2d, d2h, {"h2d": 210.0, "d2h": 193.0}) == \
        pytest.approx(2 * fast)


def test_traffic_record_matches_the_dominant_kernel_as_it_is():
    """profiles/traffic.txt holds the ncu DRAM traffic of the step's dominant
    kernel under that kernel's source hash; the bench reports it only while
    the hash matches.  A changed chain generator or common header shows here,
    before a GPU run, as a record to capture again."""
    import workloads as W
    spec, dt = W.random_chain(32, 5)

    class Item:
        kernel = ("chain", spec, (W.FLAT_SIZES[-1],), dt)
    name = f"flat_chain_L32_n{W.FLAT_SIZES[-1]}"
    assert bench.traffic_record(name, bench.kernel_source_hash(Item)) is not None
