"""batched_powerSGD_hook on the GPU against the fp64 oracle: the whole bucket
as one zero-padded square (side multiple of 4: vector path; otherwise the
element path), several replica counts and ranks, error feedback on the
padded square, the truncated output."""

import numpy as np
import pytest

import oracle
from parity_util import REL_TOL, rel
from powersgd_rank_gradient_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.mark.parametrize("numel,world,rank,dtype", [
    (1000, 2, 1, "f32"), (5000, 1, 4, "f32"), (70001, 3, 4, "f32"), (1 << 20, 2, 8, "f32"),
    ((1 << 20) + 3, 4, 2, "f32"), (25557032, 4, 1, "f32"),
    # side 1733: rows start at every offset mod 4 (the shifted-chunk pass 1)
    (3000001, 2, 8, "f32"), (3000001, 2, 8, "bf16"), (70001, 8, 4, "bf16")])
def test_batched_matches_oracle(numel, world, rank, dtype):
    from powersgd_rank_gradient_gb300 import BatchedPowerSGDState

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    st = BatchedPowerSGDState(numel, world, matrix_approximation_rank=rank, start_powerSGD_iter=1,
                              grad_dtype=tdt, device=DEV)
    ref = oracle.BatchedPowerSGDOracle(numel=numel, world_size=world, matrix_approximation_rank=rank,
                                       start_powerSGD_iter=1)
    assert st.side == ref.side and st.error_numel() == ref.side ** 2
    draw = wl.standard_normal_np((ref.side, ref.rank), numel % 1000)
    st.set_q(0, draw, is_draw=True)
    ref.set_q_draw(draw.astype(np.float64))
    rng = np.random.default_rng(numel)
    for step in range(3):
        g = [torch.from_numpy((rng.standard_normal(numel) * 1e-3).astype(np.float32)).to(tdt)
             for _ in range(world)]
        out = st.step([x.to(DEV) for x in g])
        assert not st.status()
        # the oracle sees the same (bf16-rounded) values, widened to float64
        _, exp = ref.step([x.double().numpy() for x in g])
        assert rel(out.double().cpu().numpy(), exp) <= REL_TOL, f"step {step}"
        if step >= 1:
            for w in range(world):
                e = st.get_error(w).double().cpu().numpy()
                assert rel(e, ref.error_of(w).reshape(-1)) <= REL_TOL, f"step {step} error {w}"
            p = st.get_p(0).double().numpy()
            assert np.abs(p.T @ p - np.eye(ref.rank)).max() <= 1e-4
    before, after, _ = st.stats()
    assert before == numel and after == 2 * ref.side * ref.rank
    st.close()
