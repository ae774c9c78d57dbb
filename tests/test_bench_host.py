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


def test_mufu_count_of_a_chain():
    # exp: one ex2; sigmoid: one ex2 and one rcp; the prologue, scale
    # constants and the other ops use no special-function unit
    assert bench.mufu_per_element("shuffle:4;exp") == 1
    assert bench.mufu_per_element("relu;sigmoid") == 2
    assert bench.mufu_per_element("exp;sigmoid;relu;mul") == 3
    assert bench.mufu_per_element("cast:f32;scale:0.5;add;mul") == 0


def test_cpu_all_cores_sample_uses_every_core():
    b, t, threads, desc = bench.cpu_sample_all_cores(4096)
    assert b > 0 and t > 0 and threads == (os.cpu_count() or 1) and "slices" in desc
