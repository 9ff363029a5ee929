"""Planted mistakes in the oracle must be caught by its pins.

Each test swaps one piece of the fp64 oracle (on the CPU, through
monkeypatch) for a plausible wrong version and checks that at least one pin
of ``test_oracle_pins`` then fails.  This shows the pins constrain the oracle
rather than restate it.
"""

import math

import numpy as np
import pytest

import oracle.powersgd_oracle as po
import test_oracle_pins as pins


def _any_fails(*checks):
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def _gs_eps_on_entries(matrix, epsilon):
    a = np.array(matrix, dtype=np.float64, copy=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        for i in range(a.shape[1]):
            a[:, i] = (a[:, i] + epsilon) / math.sqrt(float(np.dot(a[:, i], a[:, i])))
            for j in range(i + 1, a.shape[1]):
                a[:, j] = a[:, j] - np.dot(a[:, i], a[:, j]) * a[:, i]
    return a


def _gs_no_eps(matrix, epsilon):
    return _ORIG_GS(matrix, 0.0)


def _gs_normalise_only(matrix, epsilon):
    a = np.array(matrix, dtype=np.float64, copy=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        for i in range(a.shape[1]):
            a[:, i] = a[:, i] / (np.linalg.norm(a[:, i]) + epsilon)
    return a


def _gs_projection_sign(matrix, epsilon):
    a = np.array(matrix, dtype=np.float64, copy=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        for i in range(a.shape[1]):
            a[:, i] = a[:, i] / (np.linalg.norm(a[:, i]) + epsilon)
            for j in range(i + 1, a.shape[1]):
                a[:, j] = a[:, j] + np.dot(a[:, i], a[:, j]) * a[:, i]
    return a


_ORIG_GS = po.orthogonalize


@pytest.mark.parametrize("bad_gs", [_gs_eps_on_entries, _gs_no_eps, _gs_normalise_only,
                                    _gs_projection_sign])
def test_wrong_gram_schmidt_is_caught(monkeypatch, bad_gs):
    monkeypatch.setattr(po, "orthogonalize", bad_gs)
    monkeypatch.setattr(pins, "orthogonalize", bad_gs)
    assert _any_fails(pins.check_gs_golden, pins.check_gs_is_qr, pins.check_zero_columns_eps,
                      pins.check_pythagoras)


def test_sum_instead_of_mean_is_caught(monkeypatch):
    def allreduce_sum(arrays):
        acc = np.zeros_like(np.asarray(arrays[0], dtype=np.float64))
        for a in arrays:
            acc = acc + a
        return acc
    monkeypatch.setattr(po, "allreduce_mean", allreduce_sum)
    assert _any_fails(pins.check_2x2_golden)
    assert _any_fails(pins.check_replica_mean_linearity)


def test_transposed_q_projection_is_caught(monkeypatch):
    # M P instead of M^T P; it only type-checks on square matrices.
    monkeypatch.setattr(po, "compute_q",
                        lambda m, p: m @ p if m.shape[0] == m.shape[1] else m.T @ p)
    assert _any_fails(pins.check_pythagoras)


def test_transposed_p_projection_is_caught(monkeypatch):
    monkeypatch.setattr(po, "compute_p",
                        lambda m, q: m.T @ q if m.shape[0] == m.shape[1] else m @ q)
    assert _any_fails(pins.check_pythagoras, pins.check_svd_convergence)


def test_missing_error_feedback_is_caught(monkeypatch):
    class NoEF(po.PowerSGDOracle):
        def step(self, grads, inv_loss_scale=1.0):
            self.error.clear()
            return super().step(grads, inv_loss_scale)
    assert _any_fails(lambda: pins.check_2x2_golden(NoEF))


def test_wrong_decompression_is_caught(monkeypatch):
    monkeypatch.setattr(po, "decompress", lambda p, q: p @ (q / np.maximum(1.0, np.abs(q).max())).T)
    assert _any_fails(pins.check_2x2_golden, pins.check_rank_r_exact)


def test_non_strict_gate_is_caught(monkeypatch):
    orig = po.plan_bucket

    def plan_le(shapes, r, mcr):
        plans = orig(shapes, r, mcr)
        for p in plans:
            if len(p.shape) >= 2 and p.rows > 0 and p.cols > 0 and \
                    (p.rows + p.cols) * r * mcr <= p.rows * p.cols and not p.compressed:
                p.compressed = True
                p.rank = min(r, p.rows, p.cols)
        return plans
    monkeypatch.setattr(pins, "plan_bucket", plan_le)
    assert _any_fails(pins.check_gate_golden)


def test_vectors_compressed_is_caught(monkeypatch):
    orig = po.plan_bucket

    def plan_vectors(shapes, r, mcr):
        plans = orig(shapes, r, mcr)
        for p in plans:
            if len(p.shape) == 1 and p.numel > 2 * r * mcr:
                p.compressed = True
        return plans
    monkeypatch.setattr(pins, "plan_bucket", plan_vectors)
    assert _any_fails(pins.check_gate_golden)


def test_no_skip_on_nonfinite_is_caught(monkeypatch):
    monkeypatch.setattr(po.np, "isfinite", lambda x: np.ones_like(x, dtype=bool))
    assert _any_fails(pins.check_nonfinite_skip)
