"""CPU checks of the C ABI: the library loads, exports every symbol the header
declares, and its host-only planner agrees with the gate of the pages."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import plan_bucket
from powersgd_rank_gradient_gb300 import _lib, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "psgd.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psgd_[a-z_]+)\s*\(", text)))


def test_header_symbols_are_exported():
    L = _lib.lib()
    names = _declared()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), n
    assert sorted(_lib.EXPORTS) == names


def test_loaded_library_matches_its_sources():
    """The library carries the hash of the sources, header, flags and compiler
    it was built from; the loaded one must match the files in this tree (no
    stale binary)."""
    from powersgd_rank_gradient_gb300 import build

    bid = _lib.lib().psgd_build_id().decode()
    assert bid == "psgd-source-hash:" + build.source_hash()
    assert build.library_hash() == build.source_hash()


def test_plan_matches_gate_golden():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "gate_cases.json")))
    for case in g["cases"]:
        comp, ranks, rows, cols = _lib.plan([case["shape"]], case["rank"], case["mcr"])
        assert comp[0] == int(case["compressed"]), case
        assert ranks[0] == case["rank_eff"], case


@pytest.mark.parametrize("name,fn", [("resnet50", workloads.resnet50_shapes),
                                     ("bert-large", workloads.bert_large_shapes),
                                     ("gpt2-xl", workloads.gpt2_xl_shapes)])
def test_plan_matches_oracle_on_buckets(name, fn):
    w = workloads.WORKLOADS[name]
    shapes = fn()
    comp, ranks, rows, cols = _lib.plan(shapes, w["rank"], w["mcr"])
    ref = plan_bucket(shapes, w["rank"], w["mcr"])
    assert comp == [int(p.compressed) for p in ref]
    assert ranks == [p.rank for p in ref]
    assert rows == [p.rows for p in ref]
    assert cols == [p.cols for p in ref]


def test_plan_random_shapes_and_rates():
    rng = np.random.default_rng(0)
    for _ in range(200):
        nd = int(rng.integers(0, 5))
        shape = tuple(int(x) for x in rng.integers(0, 40, size=nd))
        rank = int(rng.integers(1, 33))
        mcr = float(rng.choice([0.0, 0.25, 0.5, 1.0, 1.5, 2.0, 4.0]))
        comp, ranks, rows, cols = _lib.plan([shape], rank, mcr)
        ref = plan_bucket([shape], rank, mcr)[0]
        assert comp[0] == int(ref.compressed), (shape, rank, mcr)
        assert ranks[0] == ref.rank


def test_plan_rejects_bad_arguments():
    L = _lib.lib()
    d, n = _lib.shape_arrays([(4, 4)])
    assert L.psgd_plan(d, n, 1, 0, 2.0, None, None, None, None) == _lib.PSGD_EINVAL
    assert b"rank" in L.psgd_last_error()
    assert L.psgd_plan(d, n, 1, 33, 2.0, None, None, None, None) == _lib.PSGD_EINVAL
    assert L.psgd_plan(d, n, 1, 1, -1.0, None, None, None, None) == _lib.PSGD_EINVAL
    assert L.psgd_plan(d, n, 1, 1, float("nan"), None, None, None, None) == _lib.PSGD_EINVAL
    bad = (ctypes.c_int64 * 2)(-1, 4)
    assert L.psgd_plan(bad, n, 1, 1, 2.0, None, None, None, None) == _lib.PSGD_EINVAL
    assert L.psgd_plan(d, n, -1, 1, 2.0, None, None, None, None) == _lib.PSGD_EINVAL


def test_null_state_calls_fail_cleanly():
    L = _lib.lib()
    assert L.psgd_step(None, None, None, 1.0, None) == _lib.PSGD_EINVAL
    assert L.psgd_get_stats(None, None, None, None) == _lib.PSGD_EINVAL
    assert L.psgd_error_numel(None) == 0
    assert L.psgd_workspace_bytes(None) == 0
    L.psgd_state_destroy(None)


def test_group_rejects_bad_arguments():
    """Bucket-group argument checks run before any CUDA call."""
    L = _lib.lib()
    d, n = _lib.shape_arrays([(4, 4)])
    counts = (ctypes.c_int32 * 1)(1)
    out = ctypes.c_void_p()

    def create(nb, cnt, n_streams):
        return L.psgd_group_create(nb, cnt, d, n, 1, 1, 0, 2.0, 1, 1, 0.0, 0, 0, _lib.PSGD_F32, n_streams, 0,
                                   ctypes.byref(out))

    assert create(0, counts, 4) == _lib.PSGD_EINVAL
    assert create(1, None, 4) == _lib.PSGD_EINVAL
    assert create(1, counts, 0) == _lib.PSGD_EINVAL
    assert create(1, counts, _lib.PSGD_MAX_GROUP_STREAMS + 1) == _lib.PSGD_EINVAL
    assert b"n_streams" in L.psgd_last_error()
    assert create(1, (ctypes.c_int32 * 1)(-1), 4) == _lib.PSGD_EINVAL
    assert not out.value
    assert L.psgd_group_step(None, 0, None, None, 1.0, None) == _lib.PSGD_EINVAL
    assert L.psgd_group_wait(None, None) == _lib.PSGD_EINVAL
    assert L.psgd_group_bucket(None, 0, ctypes.byref(out)) == _lib.PSGD_EINVAL
    assert L.psgd_group_size(None) == 0
    L.psgd_group_destroy(None)
