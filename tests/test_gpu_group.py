"""Bucket groups (overlap across buckets): per-bucket states stepped on
several CUDA streams, against the fp64 oracle run on the concatenated bucket.

The hook runs once per gradient bucket ("DDP Communication Hooks", "What Does
a Communication Hook Operate On?"); the buckets of a group are independent, so
a group over buckets B0..Bk must compute what one state over the bucket
B0 ++ ... ++ Bk computes, tensor by tensor.
"""

import numpy as np
import pytest

import oracle
from parity_util import ORTH_TOL, REL_TOL, grads_for, rel
from powersgd_rank_gradient_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"

BUCKETS = [
    [(700, 1100), (1100,), (3,), (1030, 64)],
    [(64, 3, 7, 7), (256,), (33, 8, 3, 3)],
    [(5,), (40, 2100), (17, 16), (2048, 512)],
]


def _split(flat, buckets):
    """Per-bucket slices (copied to fresh, aligned device tensors)."""
    out, off = [], 0
    for b in buckets:
        n = sum(wl.numel(s) for s in b)
        out.append(flat[off:off + n])
        off += n
    return out


def _group(n_streams, world, rank, **kw):
    from powersgd_rank_gradient_gb300 import PowerSGDGroup

    kw.setdefault("start_powerSGD_iter", 0)
    kw.setdefault("min_compression_rate", 1.0)
    return PowerSGDGroup(BUCKETS, world, matrix_approximation_rank=rank, n_streams=n_streams, device=DEV, **kw)


def _step_all(group, host_grads, order=None):
    """One training iteration: every bucket's hook, then wait; returns the
    concatenated output (float64, host)."""
    W = len(host_grads)
    per_w = [_split(h, BUCKETS) for h in host_grads]
    outs = []
    order = order or range(len(BUCKETS))
    res = [None] * len(BUCKETS)
    for b in order:
        dev = [torch.from_numpy(np.ascontiguousarray(per_w[w][b])).to(DEV) for w in range(W)]
        res[b] = (group.step(b, dev), dev)
    group.wait()
    for b in range(len(BUCKETS)):
        outs.append(res[b][0].double().cpu().numpy())
    return np.concatenate(outs)


@pytest.mark.parametrize("world,rank,streams", [(2, 4, 3), (1, 8, 2), (4, 2, 4)])
def test_group_matches_oracle_on_concatenated_bucket(world, rank, streams):
    shapes = [s for b in BUCKETS for s in b]
    g = _group(streams, world, rank)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=world, matrix_approximation_rank=rank,
                                start_powerSGD_iter=0, min_compression_rate=1.0)
    # inject the draws: the group's bucket-local tensor t is the oracle's
    # tensor (first index of its bucket) + t
    first = np.cumsum([0] + [len(b) for b in BUCKETS])
    for bi, view in enumerate(g.buckets):
        for t in range(len(BUCKETS[bi])):
            info = view.tensor_info(t)
            if info["compressed"]:
                draw = wl.standard_normal_np((info["cols"], info["rank"]), 900 + first[bi] + t)
                view.set_q(t, draw, is_draw=True)
                ref.set_q_draw(int(first[bi] + t), draw.astype(np.float64))
    for step in range(3):
        host = grads_for(shapes, world, step)
        got = _step_all(g, host, order=reversed(range(len(BUCKETS))))
        assert not g.status()
        _, exp = ref.step([h.astype(np.float64) for h in host])
        for p in ref.plans:
            sl = slice(p.offset, p.offset + p.numel)
            assert rel(got[sl], exp[sl]) <= REL_TOL, (step, p.index)
        for bi, view in enumerate(g.buckets):
            for w in range(world):
                e = view.get_error(w).double().cpu().numpy()
                for t in range(len(BUCKETS[bi])):
                    info = view.tensor_info(t)
                    if not info["compressed"]:
                        continue
                    po, n = info["packed_offset"], wl.numel(BUCKETS[bi][t])
                    ge = int(first[bi] + t)
                    assert rel(e[po:po + n], ref.error_of(w, ge).reshape(-1)) <= REL_TOL, (step, bi, t, w)
            for t in range(len(BUCKETS[bi])):
                if view.tensor_info(t)["compressed"]:
                    p = view.get_p(t).double().numpy()
                    assert np.abs(p.T @ p - np.eye(p.shape[1])).max() <= ORTH_TOL
    g.close()


def test_group_library_draws_equal_single_state():
    """Without injected draws the group numbers its compressed tensors across
    buckets, so its Q draws -- and so its steps -- equal one state's over the
    concatenated bucket."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = [s for b in BUCKETS for s in b]
    world, rank = 2, 4
    g = _group(4, world, rank, random_seed=1234)
    one = PowerSGDState(shapes, world, matrix_approximation_rank=rank, start_powerSGD_iter=0,
                        min_compression_rate=1.0, random_seed=1234, device=DEV)
    for step in range(2):
        host = grads_for(shapes, world, step)
        got = _step_all(g, host)
        exp = one.step([torch.from_numpy(h).to(DEV) for h in host]).double().cpu().numpy()
        off = 0
        for s in shapes:
            n = wl.numel(s)
            assert rel(got[off:off + n], exp[off:off + n]) <= REL_TOL, (step, s)
            off += n
    g.close()
    one.close()


def test_group_stream_count_is_bit_identical():
    shapes = [s for b in BUCKETS for s in b]
    outs = []
    for streams in (1, 4):
        g = _group(streams, 2, 4, random_seed=7)
        got = [_step_all(g, grads_for(shapes, 2, step)) for step in range(2)]
        outs.append(got)
        g.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_group_skip_is_per_bucket():
    """inf in one bucket skips that bucket's step only."""
    shapes = [s for b in BUCKETS for s in b]
    clean, dirty = _group(3, 2, 4, random_seed=3), _group(3, 2, 4, random_seed=3)
    h0 = grads_for(shapes, 2, 0)
    a = _step_all(clean, h0)
    b = _step_all(dirty, h0)
    assert np.array_equal(a, b)
    h1 = grads_for(shapes, 2, 1)
    bad = [x.copy() for x in h1]
    n0 = sum(wl.numel(s) for s in BUCKETS[0])
    bad[1][n0 + 5] = np.inf   # bucket 1
    a = _step_all(clean, h1)
    assert not clean.status()
    b = _step_all(dirty, bad)
    assert dirty.status()
    n1 = n0 + sum(wl.numel(s) for s in BUCKETS[1])
    assert np.array_equal(a[:n0], b[:n0]) and np.array_equal(a[n1:], b[n1:])
    # the other buckets stay in lock step with the clean group, and the
    # skipped bucket's state is still usable
    h2 = grads_for(shapes, 2, 2)
    a = _step_all(clean, h2)
    b = _step_all(dirty, h2)
    assert np.array_equal(a[:n0], b[:n0]) and np.array_equal(a[n1:], b[n1:])
    assert np.all(np.isfinite(b))
    clean.close()
    dirty.close()
