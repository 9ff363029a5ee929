"""Parity at full bucket size, in the launch configuration bench.py times.

The whole ResNet-50 (W=4, r=2), BERT-large (W=8, r=4, 1% heavy rows,
batching) and GPT-2-XL (W=2, r=8) buckets run through psgd_step for the
number of warm-started steps each configuration states (ResNet-50 5,
BERT-large 10, GPT-2-XL 5): warm-started subspace iteration with error
feedback is where fp32-versus-fp64 drift would build up, so the late steps
matter most.  Every ResNet-50 tensor, and for the two large buckets a sample
-- the embeddings, the first AND the last tensor of every other matrix shape
(the first and the last layer) and a bias vector -- is checked against the
fp64 oracle run on that tensor alone, every step: the tensors of a bucket are
independent, so the one-tensor oracle is the full oracle restricted to that
tensor.
"""

import numpy as np
import pytest

import oracle
from parity_util import ORTH_TOL, REL_TOL, rel
from powersgd_rank_gradient_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _sample(shapes, n_vectors=1):
    """Indices of the first and the last tensor of every distinct >=2-D shape
    (the first and the deepest layer), plus vectors."""
    first, last = {}, {}
    picks = []
    vec = 0
    for t, s in enumerate(shapes):
        if len(s) >= 2:
            first.setdefault(s, t)
            last[s] = t
        elif len(s) == 1 and vec < n_vectors and t > 10:
            picks.append(t)
            vec += 1
    picks += list(first.values()) + list(last.values())
    return sorted(set(picks))


@pytest.mark.parametrize("name,steps", [("resnet50", 5), ("bert-large", 10), ("gpt2-xl", 5)])
def test_fullsize_bucket_sampled_tensors(name, steps):
    from powersgd_rank_gradient_gb300 import PowerSGDState

    w = wl.WORKLOADS[name]
    shapes = w["shapes"]()
    W, r = w["world_size"], w["rank"]
    st = PowerSGDState(shapes, W, matrix_approximation_rank=r, start_powerSGD_iter=0,
                       min_compression_rate=w["mcr"],
                       batch_tensors_with_same_shape=w["batch_same_shape"], device=DEV)
    # ResNet-50 is small enough to check every tensor
    picks = list(range(len(shapes))) if name == "resnet50" else _sample(shapes)
    offsets = np.cumsum([0] + [wl.numel(s) for s in shapes])
    refs = {}
    for t in picks:
        info = st.tensor_info(t)
        ref = oracle.PowerSGDOracle(shapes=[shapes[t]], world_size=W, matrix_approximation_rank=r,
                                    start_powerSGD_iter=0, min_compression_rate=w["mcr"])
        if info["compressed"]:
            draw = wl.standard_normal_np((info["cols"], info["rank"]), 7000 + t)
            st.set_q(t, draw, is_draw=True)
            ref.set_q_draw(0, draw.astype(np.float64))
        refs[t] = ref
    out = torch.empty(st.numel, dtype=torch.float32, device=DEV)
    for step in range(steps):
        grads = [wl.gaussian_bucket_torch(shapes, w["std"], wl.replica_seed(k, step), DEV,
                                          heavy_fraction=w["heavy"]) for k in range(W)]
        st.step(grads, out=out)
        assert not st.status()
        errs = [st.get_error(k) for k in range(W)]
        for t in picks:
            lo, hi = int(offsets[t]), int(offsets[t + 1])
            host = [g[lo:hi].double().cpu().numpy() for g in grads]
            _, exp = refs[t].step(host)
            got = out[lo:hi].double().cpu().numpy()
            r_out = rel(got, exp)
            assert r_out <= REL_TOL, f"{name} step {step} tensor {t} {shapes[t]}: out {r_out:.3e}"
            info = st.tensor_info(t)
            if not info["compressed"]:
                continue
            po, n = info["packed_offset"], hi - lo
            for k in range(W):
                e = errs[k][po:po + n].double().cpu().numpy()
                r_e = rel(e, refs[t].error_of(k, 0).reshape(-1))
                assert r_e <= REL_TOL, f"{name} step {step} tensor {t}: error[{k}] {r_e:.3e}"
            p = st.get_p(t).double().numpy()
            orth = np.abs(p.T @ p - np.eye(info["rank"])).max()
            assert orth <= ORTH_TOL, f"{name} step {step} tensor {t}: |P^T P - I| {orth:.3e}"
        del grads
    st.close()
    torch.cuda.empty_cache()
