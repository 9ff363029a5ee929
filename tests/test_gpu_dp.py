"""The data-parallel split on the GPU: two processes, one replica each, on the
one available GPU, exchanging through gloo (host copies) between the
library's three stages, against the single-process oracle with W = 2.

"PowerSGD Hooks", powerSGD_hook steps 2, 3.3 and 3.6: the uncompressed batch,
the Ps and the Qs are allreduced (a mean) across the workers.  Each process
runs its own CUDA context; its kernels never wait on the other process (the
exchange happens on the host between the stages).  Compared per tensor:
the output (the same on both ranks), each rank's own residual, and P^T P.
"""

import os
import socket

import numpy as np
import pytest

from parity_util import ORTH_TOL, REL_TOL, rel

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402
from powersgd_rank_gradient_gb300 import workloads as wl  # noqa: E402

pytestmark = pytest.mark.gpu

MIXED = [(700, 1100), (1100,), (3,), (1030, 64), (64, 3, 7, 7), (256,),
         (33, 8, 3, 3), (5,), (40, 2100), (17, 16)]
ALIGNED = [(640, 1024), (512,), (1032, 512), (96, 4096)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grads(shapes, step, world, inf_at, scale):
    # a GradScaler-scaled bucket holds N(0, 1e-3) gradients times the scale
    std = 1.0 if scale == 1.0 else 1e-3
    gs = [(wl.gaussian_bucket_np(shapes, std, wl.replica_seed(w, step)) * np.float32(scale))
          for w in range(world)]
    if inf_at is not None and step == inf_at[0]:
        gs[inf_at[1]][inf_at[2]] = np.inf
    return gs


def _to_dtype(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype])


def _worker(rank_id, world, port, cfg, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank_id, world_size=world)
    try:
        from powersgd_rank_gradient_gb300 import DataParallelPowerSGDState, dp_powerSGD_hook

        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        shapes = cfg["shapes"]
        st = DataParallelPowerSGDState(shapes, matrix_approximation_rank=cfg["rank"],
                                       start_powerSGD_iter=cfg["start"], min_compression_rate=1.0,
                                       use_error_feedback=cfg["ef"],
                                       orthogonalization_epsilon=cfg["eps"],
                                       grad_dtype={"f32": torch.float32, "f16": torch.float16,
                                                   "bf16": torch.bfloat16}[cfg["dtype"]], device=dev)
        for t, d in cfg["draws"].items():
            st.set_q(t, d, is_draw=True)
        res = []
        for step in range(cfg["steps"]):
            host = _grads(shapes, step, world, cfg["inf_at"], cfg["scale"])[rank_id]
            g = _to_dtype(host, cfg["dtype"]).to(dev)
            out = torch.empty(st.numel, dtype=torch.float32, device=dev)
            dp_powerSGD_hook(st, g, out=out, inv_loss_scale=1.0 / cfg["scale"])
            skipped = st.status()
            err = st.get_error(0).cpu().numpy().copy() if cfg["ef"] else None
            ps = {t: st.get_p(t).numpy().copy() for t in cfg["draws"]}
            res.append((out.cpu().numpy().copy(), skipped, err, ps))
        st.close()
        results[rank_id] = res
    finally:
        dist.destroy_process_group()


def _run(shapes, rank, steps, start=0, ef=True, eps=0.0, dtype="f32", inf_at=None, scale=1.0, world=2):
    plans = oracle.plan_bucket(shapes, rank, 1.0)
    draws = {pl.index: wl.standard_normal_np((pl.cols, pl.rank), 900 + pl.index)
             for pl in plans if pl.compressed}
    cfg = dict(shapes=shapes, rank=rank, steps=steps, start=start, ef=ef, eps=eps, dtype=dtype,
               inf_at=inf_at, scale=scale, draws=draws)
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, port, cfg, results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=world, matrix_approximation_rank=rank,
                                start_powerSGD_iter=start, min_compression_rate=1.0,
                                use_error_feedback=ef, orthogonalization_epsilon=eps)
    for t, d in draws.items():
        ref.set_q_draw(t, d.astype(np.float64))
    for step in range(steps):
        host = _grads(shapes, step, world, inf_at, scale)
        # the oracle sees the values the GPU sees: the 16-bit rounding of the inputs
        host = [_to_dtype(h, dtype).double().numpy() for h in host]
        status, exp = ref.step(host, inv_loss_scale=1.0 / scale)
        for r in range(world):
            out, skipped, err, ps = got[r][step]
            assert skipped == (status == oracle.SKIPPED), f"rank {r} step {step}"
            if skipped:
                continue
            for pl in ref.plans:
                sl = slice(pl.offset, pl.offset + pl.numel)
                ro = rel(out[sl].astype(np.float64), exp[sl])
                assert ro <= REL_TOL, f"rank {r} step {step} tensor {pl.index}: out {ro:.3e}"
                if not pl.compressed or step < start:
                    continue
                if ef:
                    info_off = sum(p.numel for p in ref.plans[:pl.index] if p.compressed)
                    e = err[info_off:info_off + pl.numel].astype(np.float64)
                    re_ = rel(e, ref.error_of(r, pl.index).reshape(-1))
                    assert re_ <= REL_TOL, f"rank {r} step {step} tensor {pl.index}: error {re_:.3e}"
                p = ps[pl.index].astype(np.float64)
                orth = np.abs(p.T @ p - np.eye(pl.rank)).max()
                assert orth <= ORTH_TOL, f"rank {r} step {step} tensor {pl.index}: |P^T P - I| {orth:.3e}"


@pytest.mark.parametrize("rank", [1, 4, 8])
def test_dp_two_processes_mixed_bucket(rank):
    _run(MIXED, rank, 3)


@pytest.mark.parametrize("rank", [16, 32])
def test_dp_two_processes_high_ranks(rank):
    _run(ALIGNED, rank, 3)


def test_dp_vanilla_then_compressed_no_ef_eps():
    _run(MIXED, 4, 3, start=1, ef=False, eps=1e-8)


def test_dp_bf16_buckets():
    _run(MIXED, 4, 3, dtype="bf16")


def test_dp_fp16_scaled_inf_on_one_rank_skips_both():
    # GradScaler-style fp16 x 65536; rank 1 holds an inf at step 1: both
    # ranks skip that step and the next one matches the oracle
    _run(MIXED, 4, 3, dtype="f16", inf_at=(1, 1, 12345), scale=65536.0)
