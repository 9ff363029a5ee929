"""Helpers for the GPU-vs-oracle parity tests: run the CUDA library and the
fp64 oracle on the same seeded inputs and compare every step, tensor by
tensor.

Tolerances: relative Frobenius error <= 1e-4 on the decompressed output and on
every replica's error-feedback residual, and max |P^T P - I| <= 1e-4 on the
orthogonalised P, per tensor (so small tensors cannot hide behind big ones).
Uncompressed tensors (a plain mean) are compared the same way.
"""

from __future__ import annotations

import numpy as np

import oracle
from powersgd_rank_gradient_gb300 import workloads

REL_TOL = 1e-4
ORTH_TOL = 1e-4


def rel(a, b):
    nb = np.linalg.norm(b)
    na = np.linalg.norm(a - b)
    if nb == 0:
        return na
    return na / nb


class Pair:
    """A GPU state and an oracle with the same configuration."""

    def __init__(self, shapes, world, rank, device, grad_dtype=None, inject_draws=True, draw_seed=1,
                 **kw):
        import torch

        from powersgd_rank_gradient_gb300 import PowerSGDState

        self.torch = torch
        self.shapes = shapes
        self.world = world
        self.kw = kw
        self.gpu = PowerSGDState(shapes, world, matrix_approximation_rank=rank, device=device,
                                 grad_dtype=grad_dtype or torch.float32, **kw)
        self.ref = oracle.PowerSGDOracle(shapes=shapes, world_size=world,
                                         matrix_approximation_rank=rank, **kw)
        self.device = device
        self.draw_seed = draw_seed
        if inject_draws:
            self.inject_draws()

    def inject_draws(self, seed=None):
        seed = self.draw_seed if seed is None else seed
        for t, plan in enumerate(self.ref.plans):
            if plan.compressed:
                draw = workloads.standard_normal_np((plan.cols, plan.rank), seed * 1000 + t)
                self.gpu.set_q(t, draw, is_draw=True)
                self.ref.set_q_draw(t, draw.astype(np.float64))

    def step(self, host_grads, inv_loss_scale=1.0):
        torch = self.torch
        dev_grads = [torch.from_numpy(np.ascontiguousarray(h)).to(self.device) for h in host_grads]
        out = self.gpu.step(dev_grads, inv_loss_scale=inv_loss_scale)
        skipped = self.gpu.status()
        status, exp = self.ref.step([h for h in host_grads], inv_loss_scale=inv_loss_scale)
        return skipped, status, out, exp

    def compare(self, out, exp, check_error=True, check_factors=True, label=""):
        """Per-tensor comparison of the last step.  Returns the worst errors."""
        got = out.double().cpu().numpy()
        worst = {"out": 0.0, "err": 0.0, "orth": 0.0}
        errs = None
        if check_error and self.ref.use_error_feedback:
            errs = [self.gpu.get_error(w).double().cpu().numpy() for w in range(self.world)]
        for plan in self.ref.plans:
            sl = slice(plan.offset, plan.offset + plan.numel)
            r = rel(got[sl], exp[sl])
            worst["out"] = max(worst["out"], r)
            assert r <= REL_TOL, f"{label} tensor {plan.index} {plan.shape}: out rel {r:.3e}"
            if not plan.compressed:
                continue
            if errs is not None and self.ref.iter > self.ref.start_powerSGD_iter:
                info = self.gpu.tensor_info(plan.index)
                po = info["packed_offset"]
                for w in range(self.world):
                    e_gpu = errs[w][po:po + plan.numel]
                    e_ref = self.ref.error_of(w, plan.index).reshape(-1)
                    r = rel(e_gpu, e_ref)
                    worst["err"] = max(worst["err"], r)
                    assert r <= REL_TOL, f"{label} tensor {plan.index}: error[{w}] rel {r:.3e}"
            if check_factors and plan.index in self.ref.last_p:
                p = self.gpu.get_p(plan.index).double().numpy()
                orth = np.abs(p.T @ p - np.eye(plan.rank)).max()
                worst["orth"] = max(worst["orth"], orth)
                assert orth <= ORTH_TOL, f"{label} tensor {plan.index}: |P^T P - I| {orth:.3e}"
        return worst

    def close(self):
        self.gpu.close()


def grads_for(shapes, world, step, std=1.0, heavy=0.0, dtype=np.float32, scale=1.0):
    out = []
    for w in range(world):
        g = workloads.gaussian_bucket_np(shapes, std, workloads.replica_seed(w, step),
                                         heavy_fraction=heavy)
        out.append((g * np.float32(scale)).astype(dtype))
    return out
