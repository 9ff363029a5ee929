"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each ``check_*`` function raises AssertionError on a mismatch.  The tests call
them on the oracle as written; ``tests/test_oracle_mutations.py`` calls the
same checks on oracles with a planted mistake and expects them to fail.

Sources (DDP Communication Hooks, PyTorch 1.11 docs unless stated):
* "PowerSGD State" item 3 (gate), item 4 (epsilon);
* "PowerSGD Hooks", powerSGD_hook steps 1-3.7 and the vanilla-allreduce note;
* "Default Communication Hooks", allreduce_hook (mean);
* torch.cuda.amp "GradScaler" (unscale, inf/NaN check, skipped step).
"""

import copy
import json
import os

import numpy as np
import pytest

import oracle
from oracle import PowerSGDOracle, orthogonalize, plan_bucket
from powersgd_rank_gradient_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


# --------------------------------------------------------------------------
# Gate and views (hand-worked table; bucket counts from the shape lists)
# --------------------------------------------------------------------------
def check_gate_golden():
    g = _load("gate_cases.json")
    for case in g["cases"]:
        plan = plan_bucket([tuple(case["shape"])], case["rank"], case["mcr"])[0]
        assert plan.compressed == case["compressed"], case
        assert plan.rank == case["rank_eff"], case
    shape_fns = {"resnet50": workloads.resnet50_shapes,
                 "bert-large": workloads.bert_large_shapes,
                 "gpt2-xl": workloads.gpt2_xl_shapes}
    for name, exp in g["bucket_counts"].items():
        if name == "why":
            continue
        plans = plan_bucket(shape_fns[name](), exp["rank"], exp["mcr"])
        assert len(plans) == exp["tensors"], name
        assert sum(p.compressed for p in plans) == exp["compressed"], name
        assert sum(p.numel for p in plans if not p.compressed) == exp["uncompressed_numel"], name
        assert sum(p.numel for p in plans if p.compressed) == exp["compressed_numel"], name


def test_gate_golden():
    check_gate_golden()


def test_views_offsets():
    plans = plan_bucket([(3, 2, 2), (5,), (4, 4)], 1, 0.5)
    assert [(p.offset, p.numel) for p in plans] == [(0, 12), (12, 5), (17, 16)]
    assert (plans[0].rows, plans[0].cols) == (3, 4)
    assert not plans[1].compressed


# --------------------------------------------------------------------------
# Gram-Schmidt
# --------------------------------------------------------------------------
def check_gs_golden():
    for case in _load("gram_schmidt_cases.json")["cases"]:
        out = orthogonalize(np.array(case["input"]), case["eps"])
        if case["expected"] == "nan":
            assert np.isnan(out).all(), case["name"]
        else:
            np.testing.assert_allclose(out, np.array(case["expected"]), rtol=0, atol=1e-14,
                                       err_msg=case["name"])


def test_gs_golden():
    check_gs_golden()


def check_gs_is_qr():
    """eps = 0: Gram-Schmidt equals the Q factor of a Householder QR (LAPACK)
    with the signs fixed so that diag(R) > 0."""
    rng = np.random.default_rng(7)
    for n, r in [(5, 1), (8, 3), (64, 8), (300, 32), (33, 7)]:
        a = rng.standard_normal((n, r))
        q, rr = np.linalg.qr(a)
        q = q * np.sign(np.diag(rr))[None, :]
        out = orthogonalize(a, 0.0)
        np.testing.assert_allclose(out, q, rtol=0, atol=1e-11)
        np.testing.assert_allclose(out.T @ out, np.eye(r), atol=1e-12)


def test_gs_is_qr():
    check_gs_is_qr()


def test_gs_eps_small_effect():
    """eps > 0 moves the result by O(eps / ||column||) only."""
    rng = np.random.default_rng(8)
    a = rng.standard_normal((50, 4))
    d = np.abs(orthogonalize(a, 1e-8) - orthogonalize(a, 0.0)).max()
    assert d < 1e-8


# --------------------------------------------------------------------------
# The hand-worked 2x2, two-replica, two-step example
# --------------------------------------------------------------------------
def check_2x2_golden(factory=PowerSGDOracle):
    g = _load("powersgd_2x2_two_replicas.json")
    c = g["config"]
    o = factory(shapes=[tuple(s) for s in c["shapes"]], world_size=c["world_size"],
                matrix_approximation_rank=c["matrix_approximation_rank"],
                start_powerSGD_iter=c["start_powerSGD_iter"],
                min_compression_rate=c["min_compression_rate"],
                use_error_feedback=c["use_error_feedback"], warm_start=c["warm_start"],
                orthogonalization_epsilon=c["orthogonalization_epsilon"])
    o.set_q_draw(0, np.array(g["q_draw"]))
    for st in g["steps"]:
        status, out = o.step([np.array(x) for x in st["grads"]])
        assert status == oracle.OK
        np.testing.assert_allclose(out, st["out"], atol=1e-13)
        for w in range(2):
            np.testing.assert_allclose(o.error_of(w, 0).reshape(-1), st["error"][w], atol=1e-13)
        np.testing.assert_allclose(o.last_p[0].reshape(-1), st["p"], atol=1e-13)
        np.testing.assert_allclose(o.q[0].reshape(-1), st["q"], atol=1e-13)


def test_2x2_golden():
    check_2x2_golden()


# --------------------------------------------------------------------------
# Closed forms and invariants of one compressed step
# --------------------------------------------------------------------------
def _one_step(shape, world, rank, seed, eps=0.0, ef=True, grads=None, draw=None):
    rng = np.random.default_rng(seed)
    n, m = shape
    o = PowerSGDOracle(shapes=[shape], world_size=world, matrix_approximation_rank=rank,
                       start_powerSGD_iter=0, min_compression_rate=0.0,
                       use_error_feedback=ef, orthogonalization_epsilon=eps)
    if grads is None:
        grads = [rng.standard_normal(n * m) for _ in range(world)]
    if draw is None:
        draw = rng.standard_normal((m, o.plans[0].rank))
    o.set_q_draw(0, draw)
    status, out = o.step(grads)
    return o, grads, out


def check_rank_r_exact():
    """If the mean gradient has rank <= r and Q sees all of it, P Q^T
    reconstructs it exactly and the mean error is zero."""
    rng = np.random.default_rng(11)
    for (n, m, r, world) in [(40, 30, 3, 1), (17, 64, 4, 3), (64, 9, 2, 2)]:
        a = rng.standard_normal((n, r))
        b = rng.standard_normal((m, r))
        mbar = a @ b.T
        d = [rng.standard_normal((n, m)) for _ in range(world - 1)]
        d.append(-sum(d) if d else np.zeros((n, m)))
        grads = [(mbar + d[w]).reshape(-1) for w in range(world)]
        o, _, out = _one_step((n, m), world, r, 3, grads=grads)
        assert _rel(out.reshape(n, m), mbar) < 1e-12
        for w in range(world):
            assert _rel(o.error_of(w, 0), d[w]) < 1e-10 or np.linalg.norm(d[w]) == 0
            if np.linalg.norm(d[w]) == 0:
                assert np.abs(o.error_of(w, 0)).max() < 1e-12


def test_rank_r_exact():
    check_rank_r_exact()


def check_pythagoras():
    """P orthonormal; mean error orthogonal to P; ||Mbar||^2 = ||Mhat||^2 +
    ||ebar||^2; rank(Mhat) <= r."""
    for (n, m, r, world) in [(30, 20, 3, 2), (64, 128, 8, 4), (9, 5, 2, 1), (16, 16, 3, 2)]:
        o, grads, out = _one_step((n, m), world, r, 5 + n)
        mbar = sum(g.reshape(n, m) for g in grads) / world
        mhat = out.reshape(n, m)
        ebar = sum(o.error_of(w, 0) for w in range(world)) / world
        p = o.last_p[0]
        np.testing.assert_allclose(p.T @ p, np.eye(r), atol=1e-12)
        assert np.abs(p.T @ ebar).max() < 1e-12 * max(1.0, np.abs(mbar).max()) * n
        lhs = np.linalg.norm(mbar) ** 2
        rhs = np.linalg.norm(mhat) ** 2 + np.linalg.norm(ebar) ** 2
        assert abs(lhs - rhs) < 1e-11 * lhs
        s = np.linalg.svd(mhat, compute_uv=False)
        assert np.all(s[r:] < 1e-11 * s[0])


def test_pythagoras():
    check_pythagoras()


def check_rank1_closed_form():
    """r = 1: p = Mbar q / ||Mbar q||, q' = Mbar^T p, Mhat = p q'^T, with q the
    normalised draw and Mbar the replica mean."""
    rng = np.random.default_rng(21)
    n, m, world = 12, 7, 3
    grads = [rng.standard_normal(n * m) for _ in range(world)]
    draw = rng.standard_normal((m, 1))
    o, _, out = _one_step((n, m), world, 1, 0, grads=grads, draw=draw)
    mbar = sum(g.reshape(n, m) for g in grads) / world
    q = draw[:, 0] / np.linalg.norm(draw[:, 0])
    v = mbar @ q
    p = v / np.linalg.norm(v)
    q1 = mbar.T @ p
    np.testing.assert_allclose(out.reshape(n, m), np.outer(p, q1), atol=1e-13)
    np.testing.assert_allclose(o.q[0][:, 0], q1, atol=1e-13)


def test_rank1_closed_form():
    check_rank1_closed_form()


def check_replica_mean_linearity():
    """W replicas give the same output as one replica holding the mean, and the
    mean of the W errors equals that replica's error (the allreduce is a mean)."""
    rng = np.random.default_rng(31)
    n, m, r, world = 20, 16, 3, 4
    draw = rng.standard_normal((m, r))
    ow = PowerSGDOracle(shapes=[(n, m)], world_size=world, matrix_approximation_rank=r,
                        start_powerSGD_iter=0, min_compression_rate=0.0)
    o1 = PowerSGDOracle(shapes=[(n, m)], world_size=1, matrix_approximation_rank=r,
                        start_powerSGD_iter=0, min_compression_rate=0.0)
    ow.set_q_draw(0, draw)
    o1.set_q_draw(0, draw)
    for step in range(3):
        grads = [rng.standard_normal(n * m) for _ in range(world)]
        _, outw = ow.step(grads)
        _, out1 = o1.step([sum(grads) / world])
        np.testing.assert_allclose(outw, out1, atol=1e-12)
        ebar = sum(ow.error_of(w, 0) for w in range(world)) / world
        np.testing.assert_allclose(ebar, o1.error_of(0, 0), atol=1e-12)


def test_replica_mean_linearity():
    check_replica_mean_linearity()


# --------------------------------------------------------------------------
# Across steps
# --------------------------------------------------------------------------
def check_svd_convergence():
    """Fixed gradient, EF off, warm start on: the steps are subspace iteration,
    so span(P) converges to the top-r left singular subspace and Mhat to the
    rank-r truncated SVD (brute force with LAPACK's SVD)."""
    rng = np.random.default_rng(41)
    for (n, m, r, spectrum) in [(8, 6, 2, [9.0, 7.0, 2.0, 1.0, 0.5, 0.1]),
                                (32, 16, 3, [10.0, 8.0, 6.0] + [1.0] * 13),
                                (10, 10, 2, [5.0, 4.0, 1.0, 0.9, 0.5, 0.4, 0.3, 0.2, 0.1, 0.05])]:
        u, _ = np.linalg.qr(rng.standard_normal((n, n)))
        v, _ = np.linalg.qr(rng.standard_normal((m, m)))
        s = np.zeros((n, m))
        s[np.arange(len(spectrum)), np.arange(len(spectrum))] = spectrum
        mat = u @ s @ v.T
        o = PowerSGDOracle(shapes=[(n, m)], world_size=1, matrix_approximation_rank=r,
                           start_powerSGD_iter=0, min_compression_rate=0.0,
                           use_error_feedback=False)
        o.set_q_draw(0, rng.standard_normal((m, r)))
        uu, ss, vv = np.linalg.svd(mat)
        proj = uu[:, :r] @ uu[:, :r].T
        best = (uu[:, :r] * ss[:r]) @ vv[:r]
        dists = []
        for _ in range(30):
            _, out = o.step([mat.reshape(-1)])
            p = o.last_p[0]
            dists.append(np.linalg.norm(p @ p.T - proj))
        ratio = (spectrum[r] / spectrum[r - 1]) ** 2
        assert dists[-1] < 1e-9
        assert dists[10] < 10 * ratio ** 10 * max(dists[0], 1e-3) + 1e-12
        assert _rel(out.reshape(n, m), best) < 1e-9


def test_svd_convergence():
    check_svd_convergence()


def check_ef_telescoping():
    """Error feedback loses nothing: sum_t out_t + mean_w e_{w,T} equals
    sum_t mean_w g_{w,t}, and e_{w,t} - e_{w',t} = g_{w,t} - g_{w',t} +
    e_{w,t-1} - e_{w',t-1}."""
    rng = np.random.default_rng(51)
    shapes = [(12, 10), (7,), (6, 3, 2)]
    world = 3
    o = PowerSGDOracle(shapes=shapes, world_size=world, matrix_approximation_rank=2,
                       start_powerSGD_iter=0, min_compression_rate=0.5)
    n = o.numel
    sum_out = np.zeros(n)
    sum_mean = np.zeros(n)
    prev = {k: v.copy() for k, v in o.error.items()}
    for _ in range(6):
        grads = [rng.standard_normal(n) for _ in range(world)]
        _, out = o.step(grads)
        sum_out += out
        sum_mean += sum(grads) / world
        for plan in o.plans:
            if not plan.compressed:
                continue
            sl = slice(plan.offset, plan.offset + plan.numel)
            t = plan.index
            for w in range(1, world):
                lhs = o.error_of(w, t) - o.error_of(0, t)
                e_prev_w = prev.get((w, t), np.zeros((plan.rows, plan.cols)))
                e_prev_0 = prev.get((0, t), np.zeros((plan.rows, plan.cols)))
                rhs = ((grads[w][sl] - grads[0][sl]).reshape(plan.rows, plan.cols)
                       + e_prev_w - e_prev_0)
                np.testing.assert_allclose(lhs, rhs, atol=1e-12)
        prev = {k: v.copy() for k, v in o.error.items()}
    ebar = np.zeros(n)
    for plan in o.plans:
        if plan.compressed:
            sl = slice(plan.offset, plan.offset + plan.numel)
            ebar[sl] = sum(o.error_of(w, plan.index).reshape(-1) for w in range(world)) / world
    np.testing.assert_allclose(sum_out + ebar, sum_mean, atol=1e-11)


def test_ef_telescoping():
    check_ef_telescoping()


def check_vanilla_phase():
    """Before start_powerSGD_iter the hook is the plain mean and touches no
    state; compression starts at call number start_powerSGD_iter."""
    rng = np.random.default_rng(61)
    shapes = [(6, 5), (4,)]
    o = PowerSGDOracle(shapes=shapes, world_size=2, matrix_approximation_rank=1,
                       start_powerSGD_iter=2, min_compression_rate=0.5)
    for it in range(2):
        grads = [rng.standard_normal(34) for _ in range(2)]
        status, out = o.step(grads)
        assert status == oracle.OK
        np.testing.assert_array_equal(out, (grads[0] + grads[1]) / 2)
        assert not o.q and not o.error
    assert o.iter == 2
    o.step([rng.standard_normal(34) for _ in range(2)])
    assert 0 in o.q and (0, 0) in o.error


def test_vanilla_phase():
    check_vanilla_phase()


def check_nonfinite_skip():
    """GradScaler: a step whose (unscaled) gradients hold inf or NaN is
    skipped; the hook state is left exactly as it was."""
    rng = np.random.default_rng(71)
    o = PowerSGDOracle(shapes=[(8, 6), (3,)], world_size=2, matrix_approximation_rank=2,
                       start_powerSGD_iter=0, min_compression_rate=0.5)
    o.step([rng.standard_normal(51) for _ in range(2)])
    before = copy.deepcopy((o.q, o.error, o.last_p))
    for bad in (np.inf, -np.inf, np.nan):
        grads = [rng.standard_normal(51) for _ in range(2)]
        grads[1][rng.integers(51)] = bad
        it = o.iter
        status, out = o.step(grads)
        assert status == oracle.SKIPPED and out is None
        assert o.iter == it + 1
        after = (o.q, o.error, o.last_p)
        for d0, d1 in zip(before, after):
            assert d0.keys() == d1.keys()
            for k in d0:
                np.testing.assert_array_equal(d0[k], d1[k])


def test_nonfinite_skip():
    check_nonfinite_skip()


def check_zero_columns_eps():
    """Three all-zero columns of P (the gradient is zero along the coordinates
    the first three columns of Q live on).  eps = 1e-8 keeps them exactly zero
    with no NaN and P^T P = diag(0,0,0,1,...); eps = 0 gives NaN."""
    rng = np.random.default_rng(81)
    n, m, r = 64, 32, 8
    zero_cols = np.sort(rng.permutation(m)[:3])
    mat = rng.standard_normal((n, m))
    mat[:, zero_cols] = 0.0
    draw = rng.standard_normal((m, r))
    draw[:, :3] = 0.0
    draw[zero_cols, np.arange(3)] = 1.0
    o, _, out = _one_step((n, m), 1, r, 0, eps=1e-8, grads=[mat.reshape(-1)], draw=draw)
    p = o.last_p[0]
    assert np.all(np.isfinite(p)) and np.all(np.isfinite(out))
    assert np.all(p[:, :3] == 0.0)
    np.testing.assert_allclose(p.T @ p, np.diag([0, 0, 0, 1, 1, 1, 1, 1]), atol=1e-7)
    o0, _, out0 = _one_step((n, m), 1, r, 0, eps=0.0, grads=[mat.reshape(-1)], draw=draw)
    assert np.isnan(o0.last_p[0]).any()


def test_zero_columns_eps():
    check_zero_columns_eps()


def check_warm_vs_cold():
    """warm_start=False with the injected draw equal to the previous averaged
    Q gives the warm-start result: orthogonalising Q only multiplies it by an
    upper-triangular matrix with a positive diagonal, which leaves
    orth(M Q) unchanged (eps = 0)."""
    rng = np.random.default_rng(91)
    n, m, r = 24, 18, 3
    kw = dict(shapes=[(n, m)], world_size=2, matrix_approximation_rank=r,
              start_powerSGD_iter=0, min_compression_rate=0.0)
    warm = PowerSGDOracle(warm_start=True, **kw)
    cold = PowerSGDOracle(warm_start=False, **kw)
    draw = rng.standard_normal((m, r))
    warm.set_q_draw(0, draw)
    cold.set_q_draw(0, draw)
    for _ in range(4):
        grads = [rng.standard_normal(n * m) for _ in range(2)]
        if 0 in warm.q:
            cold.set_q_draw(0, warm.q[0])
        _, ow = warm.step(grads)
        _, oc = cold.step(grads)
        np.testing.assert_allclose(ow, oc, atol=1e-10)


def test_warm_vs_cold():
    check_warm_vs_cold()


def test_fp16_unscale():
    """fp16 gradients pre-scaled by 65536 are unscaled exactly (power of two)."""
    rng = np.random.default_rng(101)
    n, m = 16, 12
    g16 = (rng.standard_normal(n * m) * 1e-3 * 65536).astype(np.float16)
    draw = rng.standard_normal((m, 2))
    a, _, out_a = _one_step((n, m), 1, 2, 0, grads=[g16], draw=draw)
    # same step fed float64 values that are already unscaled
    o = PowerSGDOracle(shapes=[(n, m)], world_size=1, matrix_approximation_rank=2,
                       start_powerSGD_iter=0, min_compression_rate=0.0)
    o.set_q_draw(0, draw)
    _, out_b = o.step([g16.astype(np.float64) / 65536.0], inv_loss_scale=1.0)
    a2 = PowerSGDOracle(shapes=[(n, m)], world_size=1, matrix_approximation_rank=2,
                        start_powerSGD_iter=0, min_compression_rate=0.0)
    a2.set_q_draw(0, draw)
    _, out_c = a2.step([g16], inv_loss_scale=2.0 ** -16)
    np.testing.assert_array_equal(out_b, out_c)


def test_batch_flag_values():
    """batch_tensors_with_same_shape changes scheduling only."""
    rng = np.random.default_rng(111)
    shapes = [(8, 6), (8, 6), (5,), (8, 6)]
    outs = []
    for flag in (False, True):
        o = PowerSGDOracle(shapes=shapes, world_size=2, matrix_approximation_rank=2,
                           start_powerSGD_iter=0, min_compression_rate=0.5,
                           batch_tensors_with_same_shape=flag, random_seed=3)
        r2 = np.random.default_rng(5)
        outs.append([o.step([r2.standard_normal(149) for _ in range(2)])[1] for _ in range(2)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_compression_stats():
    o = PowerSGDOracle(shapes=[(8, 6), (5,)], world_size=1, matrix_approximation_rank=2,
                       min_compression_rate=0.5)
    assert o.compression_stats() == (53, (8 + 6) * 2 + 5)


# --------------------------------------------------------------------------
# The oracle's counter-based generator (for the library's own Q draws)
# --------------------------------------------------------------------------
def test_philox_known_answers():
    from oracle.philox import philox4x32_10

    for case in _load("philox_kat.json")["cases"]:
        c = [np.uint32(int(x, 16)) for x in case["counter"]]
        k = [np.uint32(int(x, 16)) for x in case["key"]]
        out = philox4x32_10(*c, *k)
        assert ["%08x" % int(x) for x in out] == case["output"]


def test_box_muller_moments():
    from oracle.philox import library_draw

    z = library_draw(4096, 8, 8, 3, 0, 1234).ravel()
    assert abs(z.mean()) < 0.02
    assert abs(z.var() - 1.0) < 0.03
    assert abs(np.mean(z ** 4) - 3.0) < 0.15   # Gaussian kurtosis


# --------------------------------------------------------------------------
# batched_powerSGD_hook
# --------------------------------------------------------------------------
def check_batched_golden():
    """N = 4 is a square: the batched hook on the 2x2 worked example's matrix
    gives the hand-worked values."""
    g = _load("powersgd_2x2_two_replicas.json")
    o = oracle.BatchedPowerSGDOracle(numel=4, world_size=2, matrix_approximation_rank=1,
                                     start_powerSGD_iter=0)
    o.set_q_draw(np.array(g["q_draw"]))
    for st in g["steps"]:
        _, out = o.step([np.array(x[:4]) for x in st["grads"]])
        np.testing.assert_allclose(out, st["out"][:4], atol=1e-13)
        for w in range(2):
            np.testing.assert_allclose(o.error_of(w).reshape(-1), st["error"][w], atol=1e-13)


def test_batched_golden():
    check_batched_golden()


@pytest.mark.parametrize("numel", [36, 37, 50, 1000])
def test_batched_is_padded_square(numel):
    """The batched hook equals the per-tensor hook run on the explicitly
    zero-padded square matrix, truncated to the bucket's length."""
    rng = np.random.default_rng(numel)
    world, rank = 3, 2
    b = oracle.BatchedPowerSGDOracle(numel=numel, world_size=world, matrix_approximation_rank=rank,
                                     start_powerSGD_iter=1)
    n = b.side
    assert n * n >= numel > (n - 1) * (n - 1)
    t = PowerSGDOracle(shapes=[(n, n)], world_size=world, matrix_approximation_rank=rank,
                       start_powerSGD_iter=1, min_compression_rate=0.0)
    draw = rng.standard_normal((n, min(rank, n)))
    b.set_q_draw(draw)
    t.set_q_draw(0, draw)
    for step in range(4):
        g = [rng.standard_normal(numel) for _ in range(world)]
        padded = []
        for x in g:
            y = np.zeros(n * n)
            y[:numel] = x
            padded.append(y)
        _, ob = b.step(g)
        _, ot = t.step(padded)
        if step == 0:
            np.testing.assert_allclose(ob, sum(g) / world, atol=1e-14)   # vanilla phase
        np.testing.assert_allclose(ob, ot[:numel], atol=1e-12)
        for w in range(world):
            np.testing.assert_allclose(b.error_of(w), t.error_of(w, 0), atol=1e-12)
