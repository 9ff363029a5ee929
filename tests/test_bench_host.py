"""Host-side pieces of bench.py that need no GPU: the committed ncu summary
is keyed to the current kernel sources, the oracle's CPU sample, and the
byte counts the roofline divides by."""

import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_committed_pass1_traffic_matches_the_kernel_sources():
    # profiles/ncu_traffic.json was captured on the sources it names; a kernel
    # change without a new capture makes the bench report traffic as null
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    assert d["src_hash"] == bench.kernel_src_hash()
    for w in ("bert-large", "gpt2-xl"):
        t = bench.ncu_traffic(w, "pass1")
        assert t is not None and t > 0
    # DRAM bytes within a few percent of the kernel's algorithmic bytes
    for case in d["small_cases"].values():
        assert 0.95 < case["pass1_traffic"] / case["pass1_algorithmic"] < 1.05


def test_oracle_sample_takes_each_shape_once_within_budget():
    spec = bench.workload_spec("bert-large")
    shapes, n = bench.oracle_sample(spec, 10_500_000)
    assert len(shapes) == len({tuple(s) for s in shapes})
    assert 0 < n <= 10_500_000
    total = 0
    for s in shapes:
        k = 1
        for dim in s:
            k *= dim
        total += k
    assert total == n
    # the first tensor of each distinct shape that fits, in bucket order
    order = [tuple(s) for s in spec["shapes"]]
    idx = [order.index(tuple(s)) for s in shapes]
    assert idx == sorted(idx)


@pytest.mark.parametrize("name,W,s_g", [("bert-large", 8, 4), ("gpt2-xl", 2, 4)])
def test_step_bytes_follow_the_design_formula(name, W, s_g):
    spec = bench.workload_spec(name)
    counts = bench.plan_counts(spec)
    sb = bench.step_bytes(spec, counts)
    assert sb["design"] > 0 and sb["survey_min"] > sb["design"]
    # pass 1 alone moves W (s_g + 8) + 4 [W >= 3] bytes per compressed element
    per_el = W * (s_g + 8) + (4 if W >= 3 else 0)
    assert sb["design"] >= per_el * counts["Nc"]
