"""The data-parallel split of the hook on CPU: two gloo ranks, one replica
each, exchange through ``dp_powerSGD_hook`` (SUM all-reduces between the
three stages) and must reproduce the single-process oracle with W = 2.

"PowerSGD Hooks", powerSGD_hook: each worker computes its own P = M_w Q and
Q = M_w^T P; the uncompressed batch (step 2), the Ps (step 3.3) and the Qs
(step 3.6) are allreduced, and the allreduce is a mean ("Default
Communication Hooks", allreduce_hook).  The stages here are a stand-in with
the oracle's own per-worker arithmetic (fp64), so what is under test is the
protocol the library's stages implement: what each stage packs for the
exchange, that the mean is the exchanged sum divided by W, and that a
non-finite input on one rank makes every rank skip the step.  The library's
kernels run the same protocol in tests/test_gpu_dp.py.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402
from powersgd_rank_gradient_gb300 import workloads as wl  # noqa: E402

SHAPES = [(40, 30), (30,), (17, 3, 2, 2), (5,), (64, 48)]


class OracleStages:
    """One worker's stages of the split step, in the oracle's arithmetic.
    begin packs [P_w of every compressed tensor | uncompressed values | flag];
    project forms P = sum / W, orthogonalises it and packs Q_w = M_w^T P;
    finish forms Q = sum / W and the output."""

    def __init__(self, shapes, world, rank, start=0, eps=0.0):
        self.plans = oracle.plan_bucket(shapes, rank, 1.0)
        self.numel = sum(p.numel for p in self.plans)
        self.world, self.start, self.eps = world, start, eps
        self.iter = 0
        self.q, self.err, self.p = {}, {}, {}
        self.draws = {}

    def begin(self, grad, out, inv_loss_scale=1.0):
        g = grad.double().numpy() * inv_loss_scale
        self.out = out
        self.vanilla = self.iter < self.start
        if self.vanilla:
            out.copy_(torch.from_numpy(g))
            return out
        self.m, parts, unc = {}, [], []
        for pl in self.plans:
            sl = slice(pl.offset, pl.offset + pl.numel)
            if not pl.compressed:
                unc.append(g[sl])
                continue
            m = g[sl].reshape(pl.rows, pl.cols) + self.err.get(pl.index, 0.0)
            self.m[pl.index] = m
            if pl.index not in self.q:
                self.q[pl.index] = oracle.orthogonalize(self.draws[pl.index], self.eps)
            parts.append(oracle.compute_p(m, self.q[pl.index]).reshape(-1))
        flag = 0.0 if np.all(np.isfinite(g)) else 1.0
        self.x = torch.from_numpy(np.concatenate(parts + unc + [np.array([flag])]))
        return self.x

    def project(self):
        if self.vanilla:
            return None
        x = self.x.numpy()
        self.skip = x[-1] != 0.0
        if self.skip:
            return None if not self.m else torch.zeros(1, dtype=torch.float64)
        off, parts = 0, []
        for pl in self.plans:
            if not pl.compressed:
                continue
            n = pl.rows * pl.rank
            p = oracle.orthogonalize(x[off:off + n].reshape(pl.rows, pl.rank) / self.world, self.eps)
            self.p[pl.index] = p
            parts.append(oracle.compute_q(self.m[pl.index], p).reshape(-1))
            off += n
        self.x_unc = x[off:-1]
        self.y = torch.from_numpy(np.concatenate(parts)) if parts else None
        return self.y

    def finish(self):
        out = self.out
        if self.vanilla:
            out.div_(self.world)
            self.status = not bool(torch.isfinite(out).all())
        elif self.skip:
            self.status = True
        else:
            y = self.y.numpy() if self.y is not None else np.zeros(0)
            off, uoff = 0, 0
            for pl in self.plans:
                sl = slice(pl.offset, pl.offset + pl.numel)
                if not pl.compressed:
                    out[sl] = torch.from_numpy(self.x_unc[uoff:uoff + pl.numel] / self.world)
                    uoff += pl.numel
                    continue
                n = pl.cols * pl.rank
                q = y[off:off + n].reshape(pl.cols, pl.rank) / self.world
                off += n
                m_hat = oracle.decompress(self.p[pl.index], q)
                out[sl] = torch.from_numpy(m_hat.reshape(-1))
                self.err[pl.index] = self.m[pl.index] - m_hat
                self.q[pl.index] = q
            self.status = False
        self.iter += 1
        return out


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grads(step, world, inf_at):
    gs = [wl.gaussian_bucket_np(SHAPES, 1.0, wl.replica_seed(w, step)).astype(np.float64) for w in range(world)]
    if inf_at is not None and step == inf_at[0]:
        gs[inf_at[1]][inf_at[2]] = np.inf
    return gs


def _draws(plans):
    return {pl.index: wl.standard_normal_np((pl.cols, pl.rank), 500 + pl.index).astype(np.float64)
            for pl in plans if pl.compressed}


def _worker(rank_id, world, port, rank, steps, start, inf_at, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank_id, world_size=world)
    try:
        from powersgd_rank_gradient_gb300.dp import dp_powerSGD_hook

        st = OracleStages(SHAPES, world, rank, start=start)
        st.draws = _draws(st.plans)
        res = []
        for step in range(steps):
            g = torch.from_numpy(_grads(step, world, inf_at)[rank_id])
            out = torch.zeros(st.numel, dtype=torch.float64)
            dp_powerSGD_hook(st, g, out=out)
            errs = {t: e.copy() for t, e in st.err.items()}
            res.append((out.numpy().copy(), st.status, errs))
        results[rank_id] = res
    finally:
        dist.destroy_process_group()


def _run(rank, steps, start=0, inf_at=None, world=2):
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, port, rank, steps, start, inf_at, results), nprocs=world,
                           join=True, start_method="spawn")
        return dict(results)


def _reference(rank, steps, start=0, inf_at=None, world=2):
    ref = oracle.PowerSGDOracle(shapes=SHAPES, world_size=world, matrix_approximation_rank=rank,
                                start_powerSGD_iter=start, min_compression_rate=1.0)
    for t, d in _draws(ref.plans).items():
        ref.set_q_draw(t, d)
    outs = []
    for step in range(steps):
        status, out = ref.step(_grads(step, world, inf_at))
        outs.append((out, status, {(w, pl.index): ref.error_of(w, pl.index).copy()
                                   for pl in ref.plans if pl.compressed for w in range(world)}))
    return outs


@pytest.mark.parametrize("rank,start", [(2, 0), (4, 0), (3, 1)])
def test_two_ranks_match_single_process_oracle(rank, start):
    steps = 3
    got = _run(rank, steps, start=start)
    exp = _reference(rank, steps, start=start)
    for step in range(steps):
        out_ref, status_ref, err_ref = exp[step]
        assert status_ref == oracle.OK
        for r in range(2):
            out, skipped, errs = got[r][step]
            assert not skipped
            np.testing.assert_allclose(out, out_ref, rtol=1e-10, atol=1e-12)
            for t, e in errs.items():
                np.testing.assert_allclose(e, err_ref[(r, t)], rtol=1e-10, atol=1e-12)


def test_nonfinite_on_one_rank_skips_every_rank():
    steps = 3
    inf_at = (1, 1, 7)          # step 1, rank 1, element 7 (inside the first matrix)
    got = _run(2, steps, inf_at=inf_at)
    exp = _reference(2, steps, inf_at=inf_at)
    assert exp[1][1] == oracle.SKIPPED
    for r in range(2):
        assert got[r][1][1] is True          # both ranks skipped step 1
        np.testing.assert_allclose(got[r][2][0], exp[2][0], rtol=1e-10, atol=1e-12)
        for t, e in got[r][2][2].items():
            np.testing.assert_allclose(e, exp[2][2][(r, t)], rtol=1e-10, atol=1e-12)
