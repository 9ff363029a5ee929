"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, every step, tensor by tensor.

Sizes are ones the oracle finishes in seconds but that still span several
column tiles and row blocks with ragged tails, unaligned tensors (odd column
counts, odd bucket offsets), every padded rank and several replica counts.
"""

import numpy as np
import pytest

from parity_util import Pair, grads_for, rel

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# A bucket with: multiple column tiles (1100, 2100 > 1024 columns), multiple
# row blocks with a ragged tail (1030 > 2 * 512 rows), an odd-sized vector in
# front of a matrix (unaligned bucket offset), an odd column count (147), a
# 4-D conv view and vectors.
MIXED = [(700, 1100), (1100,), (3,), (1030, 64), (64, 3, 7, 7), (256,),
         (33, 8, 3, 3), (5,), (40, 2100), (17, 16)]


def _run(shapes, world, rank, steps, heavy=0.0, std=1.0, label="", **kw):
    kw.setdefault("start_powerSGD_iter", 0)
    kw.setdefault("min_compression_rate", 1.0)
    pair = Pair(shapes, world, rank, DEV, **kw)
    worst = {"out": 0.0, "err": 0.0, "orth": 0.0}
    for step in range(steps):
        g = grads_for(shapes, world, step, std=std, heavy=heavy)
        skipped, status, out, exp = pair.step(g)
        assert not skipped
        w = pair.compare(out, exp, label=f"{label} step {step}")
        worst = {k: max(worst[k], w[k]) for k in worst}
    pair.close()
    return worst


def test_config1_256x512_rank1_two_steps():
    """256x512, N(0,1) from seed 0, W=1, r=1, zero error buffer, Q drawn
    N(0,1) from seed 1, eps=0, 2 warm-started steps on the same gradient."""
    from powersgd_rank_gradient_gb300 import PowerSGDState
    import oracle

    shapes = [(256, 512)]
    g = np.random.default_rng(0).standard_normal(256 * 512).astype(np.float32)
    q = np.random.default_rng(1).standard_normal((512, 1)).astype(np.float32)
    st = PowerSGDState(shapes, 1, matrix_approximation_rank=1, start_powerSGD_iter=0, device=DEV)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=1, matrix_approximation_rank=1,
                                start_powerSGD_iter=0)
    st.set_q(0, q, is_draw=True)
    ref.set_q_draw(0, q.astype(np.float64))
    for step in range(2):
        out = st.step([torch.from_numpy(g).to(DEV)])
        assert not st.status()
        _, exp = ref.step([g.astype(np.float64)])
        assert rel(out.double().cpu().numpy(), exp) <= 1e-4
        e = st.get_error(0).double().cpu().numpy()
        assert rel(e, ref.error_of(0, 0).reshape(-1)) <= 1e-4
        p = st.get_p(0).double().numpy()
        assert abs(float((p.T @ p)[0, 0]) - 1.0) <= 1e-4
        assert rel(p[:, 0], ref.last_p[0][:, 0]) <= 1e-4
        assert rel(st.get_q(0).double().numpy(), ref.q[0]) <= 1e-4
    st.close()


# 1, 2, 4, 8: the chunk-stationary pass 1 laid out for exactly W replicas;
# 3 and 5-7: the same kernel on the four- and eight-replica layouts with the
# rest unused; 9: the element kernel (any W).
@pytest.mark.parametrize("world", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_mixed_bucket_worlds(world):
    _run(MIXED, world, 4, 3, label=f"W={world}")


@pytest.mark.parametrize("rank", [1, 2, 3, 5, 8, 12, 16, 24, 32])
def test_mixed_bucket_ranks(rank):
    _run(MIXED, 2, rank, 3, min_compression_rate=0.25, label=f"r={rank}")


# Tensors whose rows are 16-byte aligned in the bucket (column counts and
# offsets multiples of 4): ranks 16 and 32 run them through the register-tiled
# pass 1.  Ragged row items (300 = 2 x 128 + 44 rows, 129 rows), ragged column
# tiles and chunks (1060 = 2 x 512 + 36 columns, 516, 36).  Every view has more
# than 32 rows and columns, so at rank 32 the residual is not rounding noise.
ALIGNED = [(300, 1060), (129, 36), (64,), (1000, 516), (48, 16, 2, 2)]


@pytest.mark.parametrize("rank", [12, 16, 24, 32])
@pytest.mark.parametrize("world,kw", [
    (1, {}),
    (3, {}),
    (8, {"heavy": 0.01, "std": 1e-3}),
    (2, {"use_error_feedback": False}),
    (2, {"orthogonalization_epsilon": 1e-8}),
], ids=["W1", "W3", "W8-heavy", "W2-noEF", "W2-eps"])
def test_aligned_bucket_high_ranks(rank, world, kw):
    _run(ALIGNED, world, rank, 3, min_compression_rate=0.25, label=f"aligned r={rank} W={world}", **kw)


@pytest.mark.parametrize("rank", [16, 32])
def test_aligned_bucket_high_ranks_cold(rank):
    """warm_start off: pass 1 projects on a fresh draw while it subtracts the
    committed factors (two different Q matrices in one pass)."""
    pair = Pair(ALIGNED, 2, rank, DEV, start_powerSGD_iter=0, min_compression_rate=0.25, warm_start=False)
    for step in range(3):
        if step > 0:
            pair.inject_draws(seed=20 + step)
        skipped, status, out, exp = pair.step(grads_for(ALIGNED, 2, step))
        assert not skipped
        pair.compare(out, exp, label=f"cold r={rank} step {step}")
    pair.close()


def test_heavy_rows_batched():
    _run(MIXED, 8, 4, 4, heavy=0.01, std=1e-3, batch_tensors_with_same_shape=True, label="heavy")


def test_vanilla_phase_then_compression():
    _run(MIXED, 3, 2, 4, start_powerSGD_iter=2, label="start=2")


def test_no_error_feedback():
    for world in (1, 2, 5):
        _run(MIXED, world, 4, 3, use_error_feedback=False, label=f"noEF W={world}")


def test_no_warm_start_fresh_draw_each_step():
    shapes = MIXED
    pair = Pair(shapes, 2, 4, DEV, start_powerSGD_iter=0, min_compression_rate=1.0,
                warm_start=False)
    for step in range(3):
        if step > 0:
            pair.inject_draws(seed=10 + step)
        skipped, status, out, exp = pair.step(grads_for(shapes, 2, step))
        pair.compare(out, exp, label=f"cold step {step}")
    pair.close()


def test_epsilon_positive():
    _run(MIXED, 2, 4, 3, orthogonalization_epsilon=1e-8, label="eps")


def test_zero_columns_with_epsilon():
    """4096x1024 gradient, r=8, eps=1e-8: the first three columns of Q live on
    coordinates where the gradient is zero, so three columns of P are exactly
    zero.  They must stay zero with no NaN, and P^T P = diag(0,0,0,1,...)."""
    import oracle

    from powersgd_rank_gradient_gb300 import PowerSGDState

    n, m, r = 4096, 1024, 8
    rng = np.random.default_rng(5)
    zero_cols = np.sort(rng.permutation(m)[:3])
    g = rng.standard_normal((n, m)).astype(np.float32)
    g[:, zero_cols] = 0.0
    draw = rng.standard_normal((m, r)).astype(np.float32)
    draw[:, :3] = 0.0
    draw[zero_cols, np.arange(3)] = 1.0
    st = PowerSGDState([(n, m)], 1, matrix_approximation_rank=r, start_powerSGD_iter=0,
                       orthogonalization_epsilon=1e-8, device=DEV)
    ref = oracle.PowerSGDOracle(shapes=[(n, m)], world_size=1, matrix_approximation_rank=r,
                                start_powerSGD_iter=0, orthogonalization_epsilon=1e-8)
    st.set_q(0, draw, is_draw=True)
    ref.set_q_draw(0, draw.astype(np.float64))
    for step in range(2):
        out = st.step([torch.from_numpy(g.reshape(-1)).to(DEV)])
        _, exp = ref.step([g.reshape(-1).astype(np.float64)])
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert rel(got, exp) <= 1e-4
        p = st.get_p(0).double().numpy()
        assert np.all(np.isfinite(p))
        assert np.all(p[:, :3] == 0.0)
        assert np.abs(p.T @ p - np.diag([0, 0, 0, 1, 1, 1, 1, 1])).max() <= 1e-4
        e = st.get_error(0).double().cpu().numpy()
        assert rel(e, ref.error_of(0, 0).reshape(-1)) <= 1e-4
    st.close()


def test_zero_p_column_eps0_gives_nan_like_oracle():
    """"PowerSGD State" item 4: with orthogonalization_epsilon = 0 an all-zero
    column of P divides zero by zero.  The first column of Q lies on a
    coordinate where the gradient is zero, so column 0 of P = M Q is exactly
    zero; the oracle's Gram-Schmidt then gives NaN in that column, and the NaN
    reaches every later column through the projections (the golden case
    "zero column, eps=0").  The GPU must give NaN in the same positions of P
    and of the output, while the uncompressed vector in the same bucket keeps
    its finite mean.  Data only: nothing traps."""
    import oracle

    from powersgd_rank_gradient_gb300 import PowerSGDState

    n, m, r = 1024, 512, 4
    shapes = [(n, m), (300,)]
    rng = np.random.default_rng(11)
    zc = 37
    g = rng.standard_normal((n, m)).astype(np.float32)
    g[:, zc] = 0.0
    vec = rng.standard_normal(300).astype(np.float32)
    bucket = np.concatenate([g.reshape(-1), vec])
    draw = rng.standard_normal((m, r)).astype(np.float32)
    draw[:, 0] = 0.0
    draw[zc, 0] = 1.0
    st = PowerSGDState(shapes, 1, matrix_approximation_rank=r, start_powerSGD_iter=0,
                       orthogonalization_epsilon=0.0, device=DEV)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=1, matrix_approximation_rank=r,
                                start_powerSGD_iter=0, orthogonalization_epsilon=0.0)
    st.set_q(0, draw, is_draw=True)
    ref.set_q_draw(0, draw.astype(np.float64))
    out = st.step([torch.from_numpy(bucket).to(DEV)])
    assert not st.status()      # the inputs are finite: the step is not skipped
    _, exp = ref.step([bucket.astype(np.float64)])
    got = out.double().cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(exp))
    assert np.isnan(exp[:n * m]).all()            # every P column is NaN -> so is P Q^T
    fin = ~np.isnan(exp)
    assert rel(got[fin], exp[fin]) <= 1e-4        # the vector's plain mean
    p_gpu = st.get_p(0).double().numpy()
    assert np.array_equal(np.isnan(p_gpu), np.isnan(ref.last_p[0]))
    st.close()


@pytest.mark.parametrize("rank,eps", [(8, 0.0), (8, 1e-8), (32, 0.0)])
def test_zero_gradient_columns_pass_through(rank, eps):
    """The second reading of the edge case with three all-zero columns: the
    gradient matrix itself has three zero columns (4096 x 1024, Q drawn at
    random).  Then Q' = M^T P has zero rows there, P Q'^T zero columns and the
    residual M - P Q'^T stays zero there, in exact arithmetic and on the GPU
    (0 * x sums to exactly 0), step after step; everything else matches the
    oracle."""
    shapes = [(4096, 1024)]
    n, m = shapes[0]
    rng = np.random.default_rng(21)
    zero_cols = np.sort(rng.permutation(m)[:3])
    pair = Pair(shapes, 1, rank, DEV, start_powerSGD_iter=0, orthogonalization_epsilon=eps)
    for step in range(3):
        g = grads_for(shapes, 1, step)[0].reshape(n, m)
        g[:, zero_cols] = 0.0
        skipped, status, out, exp = pair.step([g.reshape(-1)])
        assert not skipped
        pair.compare(out, exp, label=f"zero cols r={rank} eps={eps} step {step}")
        got = out.cpu().numpy().reshape(n, m)
        assert np.all(got[:, zero_cols] == 0.0)
        e = pair.gpu.get_error(0).cpu().numpy().reshape(n, m)
        assert np.all(e[:, zero_cols] == 0.0)
        q = pair.gpu.get_q(0).numpy()
        assert np.all(q[zero_cols, :] == 0.0)
    pair.close()


def test_fp16_scaled_with_inf_is_skipped():
    """fp16 gradients pre-scaled by 65536 and unscaled in pass 1; a step with
    one +inf is skipped with the state left bit for bit, the next clean step
    matches the oracle."""
    shapes = [(512, 768), (768,), (256, 256)]
    world = 2
    pair = Pair(shapes, world, 4, DEV, grad_dtype=torch.float16, start_powerSGD_iter=0,
                min_compression_rate=1.0)
    s = 1.0 / 65536.0
    g0 = grads_for(shapes, world, 0, std=1e-3, dtype=np.float16, scale=65536.0)
    skipped, status, out, exp = pair.step(g0, inv_loss_scale=s)
    assert not skipped
    pair.compare(out, exp, label="fp16 step 0")
    before = ([pair.gpu.get_error(w).cpu().clone() for w in range(world)],
              [pair.gpu.get_q(t).clone() for t in (0, 2)], [pair.gpu.get_p(t).clone() for t in (0, 2)])
    g1 = grads_for(shapes, world, 1, std=1e-3, dtype=np.float16, scale=65536.0)
    idx = np.random.default_rng(9).integers(g1[1].size)
    g1[1][idx] = np.float16(np.inf)
    skipped, status, out, exp = pair.step(g1, inv_loss_scale=s)
    assert skipped and status == "skipped"
    after = ([pair.gpu.get_error(w).cpu() for w in range(world)],
             [pair.gpu.get_q(t) for t in (0, 2)], [pair.gpu.get_p(t) for t in (0, 2)])
    for xs, ys in zip(before, after):
        for x, y in zip(xs, ys):
            assert torch.equal(x, y)
    g2 = grads_for(shapes, world, 2, std=1e-3, dtype=np.float16, scale=65536.0)
    skipped, status, out, exp = pair.step(g2, inv_loss_scale=s)
    assert not skipped
    pair.compare(out, exp, label="fp16 step 2")
    pair.close()


@pytest.mark.parametrize("rank", [16, 32])
def test_fp16_scaled_with_inf_high_ranks(rank):
    """The tensor-core pass 1 on fp16 gradients pre-scaled by 65536: unscaled
    in the pass, a step with one +inf is skipped with the state left bit for
    bit, the next clean step matches the oracle."""
    world = 2
    pair = Pair(ALIGNED, world, rank, DEV, grad_dtype=torch.float16, start_powerSGD_iter=0,
                min_compression_rate=0.25)
    s = 1.0 / 65536.0
    g0 = grads_for(ALIGNED, world, 0, std=1e-3, dtype=np.float16, scale=65536.0)
    skipped, status, out, exp = pair.step(g0, inv_loss_scale=s)
    assert not skipped
    pair.compare(out, exp, label=f"fp16 r={rank} step 0")
    before = ([pair.gpu.get_error(w).cpu().clone() for w in range(world)],
              [pair.gpu.get_q(t).clone() for t in (0, 3)], [pair.gpu.get_p(t).clone() for t in (0, 3)])
    g1 = grads_for(ALIGNED, world, 1, std=1e-3, dtype=np.float16, scale=65536.0)
    g1[0][7] = np.float16(np.inf)   # inside the first (aligned, compressed) tensor
    skipped, status, out, exp = pair.step(g1, inv_loss_scale=s)
    assert skipped and status == "skipped"
    after = ([pair.gpu.get_error(w).cpu() for w in range(world)],
             [pair.gpu.get_q(t) for t in (0, 3)], [pair.gpu.get_p(t) for t in (0, 3)])
    for xs, ys in zip(before, after):
        for x, y in zip(xs, ys):
            assert torch.equal(x, y)
    g2 = grads_for(ALIGNED, world, 2, std=1e-3, dtype=np.float16, scale=65536.0)
    skipped, status, out, exp = pair.step(g2, inv_loss_scale=s)
    assert not skipped
    pair.compare(out, exp, label=f"fp16 r={rank} step 2")
    pair.close()


def test_nan_in_fp32_is_skipped():
    shapes = [(300, 200), (7,)]
    pair = Pair(shapes, 2, 2, DEV, start_powerSGD_iter=0, min_compression_rate=1.0)
    skipped, _, out, exp = pair.step(grads_for(shapes, 2, 0))
    pair.compare(out, exp)
    g = grads_for(shapes, 2, 1)
    g[0][300 * 200 + 3] = np.nan      # in the uncompressed vector
    skipped, status, _, _ = pair.step(g)
    assert skipped and status == "skipped"
    skipped, _, out, exp = pair.step(grads_for(shapes, 2, 2))
    assert not skipped
    pair.compare(out, exp)
    pair.close()


def test_batch_flag_bit_identical():
    outs = []
    for flag in (False, True):
        from powersgd_rank_gradient_gb300 import PowerSGDState

        shapes = [(300, 200), (300, 200), (9,), (300, 200), (128, 64)]
        st = PowerSGDState(shapes, 2, matrix_approximation_rank=4, start_powerSGD_iter=0,
                           min_compression_rate=1.0, batch_tensors_with_same_shape=flag,
                           random_seed=7, device=DEV)
        res = []
        for step in range(3):
            g = [torch.from_numpy(x).to(DEV) for x in grads_for(shapes, 2, step)]
            res.append(st.step(g).cpu().clone())
        res.append(st.get_error(1).cpu().clone())
        outs.append(res)
        st.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_deterministic_and_out_aliases_grads0():
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = MIXED
    runs = []
    for alias in (False, True):
        st = PowerSGDState(shapes, 2, matrix_approximation_rank=4, start_powerSGD_iter=0,
                           min_compression_rate=1.0, random_seed=3, device=DEV)
        res = []
        for step in range(3):
            g = [torch.from_numpy(x).to(DEV) for x in grads_for(shapes, 2, step)]
            out = st.step(g, out=g[0] if alias else None)
            res.append(out.cpu().clone())
        runs.append(res)
        st.close()
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_error_set_get_roundtrip_and_warm_q_restore():
    """Checkpoint: copy the residuals and the warm Q of one state into a fresh
    one; both then produce the same next step (to fp32 rounding)."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = [(400, 300), (11,), (129, 64)]
    kw = dict(matrix_approximation_rank=3, start_powerSGD_iter=0, min_compression_rate=1.0,
              device=DEV)
    a = PowerSGDState(shapes, 2, random_seed=1, **kw)
    for step in range(2):
        a.step([torch.from_numpy(x).to(DEV) for x in grads_for(shapes, 2, step)])
    b = PowerSGDState(shapes, 2, random_seed=99, **kw)
    for w in range(2):
        b.set_error(w, a.get_error(w))
    for t in (0, 2):
        b.set_q(t, a.get_q(t), is_draw=False)
    for w in range(2):
        assert rel(b.get_error(w).double().cpu().numpy(), a.get_error(w).double().cpu().numpy()) < 1e-6
    g = [torch.from_numpy(x).to(DEV) for x in grads_for(shapes, 2, 5)]
    oa = a.step(g).double().cpu().numpy()
    ob = b.step(g).double().cpu().numpy()
    assert rel(ob, oa) < 1e-5
    a.close()
    b.close()


def test_library_draw_statistics():
    """The library's own standard-normal draw (no injected Q): after the first
    step P is orthonormal and the stats counters match the plan."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = [(2048, 1024)]
    st = PowerSGDState(shapes, 1, matrix_approximation_rank=8, start_powerSGD_iter=0, device=DEV,
                       random_seed=1234)
    st.step([torch.from_numpy(grads_for(shapes, 1, 0)[0]).to(DEV)])
    assert not st.status()
    p = st.get_p(0).double().numpy()
    assert np.abs(p.T @ p - np.eye(8)).max() < 1e-4
    before, after, it = st.stats()
    assert (before, after, it) == (2048 * 1024, (2048 + 1024) * 8, 1)
    st.close()


def test_invalid_arguments_are_rejected():
    from powersgd_rank_gradient_gb300 import PowerSGDState, _lib

    with pytest.raises(_lib.PsgdError):
        PowerSGDState([(4, 4)], 1, matrix_approximation_rank=0, device=DEV)
    with pytest.raises(_lib.PsgdError):
        PowerSGDState([(4, 4)], 65, device=DEV)
    st = PowerSGDState([(64, 64), (8,)], 2, matrix_approximation_rank=2, start_powerSGD_iter=0,
                       min_compression_rate=1.0, device=DEV)
    g = [torch.zeros(64 * 64 + 8, device=DEV) for _ in range(2)]
    with pytest.raises(_lib.PsgdError):
        st.step(g, out=g[1])          # out may alias only replica 0
    with pytest.raises(_lib.PsgdError):
        st.set_q(1, np.zeros((1, 1), np.float32))   # vector tensor is not compressed
    st.close()


def test_empty_and_vector_only_buckets():
    from powersgd_rank_gradient_gb300 import PowerSGDState

    st = PowerSGDState([(7,), (0, 5), (3,)], 2, start_powerSGD_iter=0, device=DEV)
    g = [torch.arange(10, dtype=torch.float32, device=DEV) * (w + 1) for w in range(2)]
    out = st.step(g)
    assert torch.allclose(out, (g[0] + g[1]) / 2)
    st.close()


@pytest.mark.parametrize("rank", [1, 2, 4, 8, 16, 32])
def test_rank_sweep_8192(rank):
    """8192 x 8192, W=1, N(0,1): three warm-started steps per rank."""
    _run([(8192, 8192)], 1, rank, 3, min_compression_rate=2.0, label=f"8192 r={rank}")


def test_step_host_matches_device_path():
    """psgd_step_host (host buffers in and out, pipelined across calls) gives
    the same bits as psgd_step on device buffers, call after call."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = MIXED
    kw = dict(matrix_approximation_rank=4, start_powerSGD_iter=1, min_compression_rate=1.0,
              random_seed=5, device=DEV)
    dev_state = PowerSGDState(shapes, 3, **kw)
    host_state = PowerSGDState(shapes, 3, **kw)
    steps = 5
    host_in = [[torch.from_numpy(x).pin_memory() for x in grads_for(shapes, 3, step)] for step in range(steps)]
    host_out = [torch.empty(dev_state.numel, dtype=torch.float32).pin_memory() for _ in range(steps)]
    # enqueue every host call back to back (the pipelined case), then compare
    for step in range(steps):
        host_state.step_host(host_in[step], host_out[step])
    torch.cuda.synchronize()
    for step in range(steps):
        out = dev_state.step([h.to(DEV) for h in host_in[step]])
        assert torch.equal(out.cpu(), host_out[step]), f"step {step}"
    dev_state.close()
    host_state.close()


@pytest.mark.parametrize("warm", [True, False])
def test_library_draw_matches_oracle_philox(warm):
    """No injected draw: the library draws Q with its Philox4x32-10 stream;
    the oracle is fed the same stream computed independently in float64."""
    import oracle
    from oracle.philox import library_draw
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = [(300, 200), (7,), (64, 3, 3, 3), (128, 96)]
    rank, seed, world = 3, 0x1234567890AB, 2
    st = PowerSGDState(shapes, world, matrix_approximation_rank=rank, start_powerSGD_iter=1,
                       min_compression_rate=1.0, warm_start=warm, random_seed=seed, device=DEV)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=world, matrix_approximation_rank=rank,
                                start_powerSGD_iter=1, min_compression_rate=1.0, warm_start=warm)
    comp = [p for p in ref.plans if p.compressed]
    rp = 4
    for step in range(4):
        if step >= 1 and (step == 1 or not warm):
            for ci, p in enumerate(comp):
                ref.set_q_draw(p.index, library_draw(p.cols, p.rank, rp, ci, step, seed))
        g = grads_for(shapes, world, step)
        out = st.step([torch.from_numpy(x).to(DEV) for x in g])
        _, exp = ref.step(g)
        got = out.double().cpu().numpy()
        for p in ref.plans:
            sl = slice(p.offset, p.offset + p.numel)
            assert rel(got[sl], exp[sl]) <= 1e-4, (step, p.index)
    st.close()


@pytest.mark.parametrize("rank", [4, 32])
@pytest.mark.parametrize("world,ef", [(1, True), (2, True), (3, False), (5, True), (8, True)])
def test_bf16_buckets(world, ef, rank):
    """16-bit (bf16) replica buckets, as the bf16 compress wrapper produces:
    the oracle is fed the same bf16 values widened to float64."""
    import oracle

    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = MIXED
    st = PowerSGDState(shapes, world, matrix_approximation_rank=rank, start_powerSGD_iter=1,
                       min_compression_rate=1.0, use_error_feedback=ef, grad_dtype=torch.bfloat16,
                       device=DEV)
    ref = oracle.PowerSGDOracle(shapes=shapes, world_size=world, matrix_approximation_rank=rank,
                                start_powerSGD_iter=1, min_compression_rate=1.0, use_error_feedback=ef)
    for t, plan in enumerate(ref.plans):
        if plan.compressed:
            from powersgd_rank_gradient_gb300 import workloads as wl
            draw = wl.standard_normal_np((plan.cols, plan.rank), 500 + t)
            st.set_q(t, draw, is_draw=True)
            ref.set_q_draw(t, draw.astype(np.float64))
    for step in range(3):
        g32 = grads_for(shapes, world, step)
        gb = [torch.from_numpy(x).to(torch.bfloat16) for x in g32]
        out = st.step([x.to(DEV) for x in gb])
        assert not st.status()
        _, exp = ref.step([x.double().numpy() for x in gb])
        got = out.double().cpu().numpy()
        for p in ref.plans:
            sl = slice(p.offset, p.offset + p.numel)
            assert rel(got[sl], exp[sl]) <= 1e-4, (step, p.index)
        if ef:
            for w in range(world):
                e = st.get_error(w).double().cpu().numpy()
                for p in ref.plans:
                    if p.compressed:
                        po = st.tensor_info(p.index)["packed_offset"]
                        assert rel(e[po:po + p.numel], ref.error_of(w, p.index).reshape(-1)) <= 1e-4
    st.close()


def test_graph_replay_bit_identical():
    """psgd_set_graph: the steady step replayed as a CUDA graph gives the same
    bits as the launch-by-launch path, through a skipped step (inf) and a
    change of output buffer (a second capture)."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = MIXED
    mk = lambda: PowerSGDState(shapes, 2, matrix_approximation_rank=4, start_powerSGD_iter=1,
                               min_compression_rate=1.0, random_seed=5, device=DEV)
    plain, graphed = mk(), mk()
    graphed.set_graph(True)
    n = plain.numel
    outs = [torch.empty(n, device=DEV), torch.empty(n, device=DEV)]
    hosts = [grads_for(shapes, 2, k) for k in range(6)]
    hosts[3] = [x.copy() for x in hosts[3]]
    hosts[3][1][7] = np.inf
    dev_sets = [[torch.empty(n, device=DEV) for _ in range(2)] for _ in range(2)]
    for step in range(6):
        ds = dev_sets[0]
        for w in range(2):
            ds[w].copy_(torch.from_numpy(hosts[step][w]))
        o = outs[1] if step == 4 else outs[0]
        a = plain.step(ds, out=o).clone()
        sa = plain.status()
        b = graphed.step(ds, out=o).clone()
        sb = graphed.status()
        assert sa == sb == (step == 3), step
        if step != 3:
            assert torch.equal(a, b), step
        for w in range(2):
            assert torch.equal(plain.get_error(w), graphed.get_error(w)), (step, w)
    # step 0 is vanilla and step 1 draws Q (no graph); step 2 captures and
    # replays, step 3 replays (skipped on the device), steps 4 and 5 change
    # the output buffer and so capture again
    assert graphed.graph_stats() == (3, 4), graphed.graph_stats()
    plain.close()
    graphed.close()


def test_profile_select_records_one_kind():
    """psgd_profile_select: only the selected kind's launches are recorded;
    psgd_profile(1) records every kind again."""
    from powersgd_rank_gradient_gb300 import PowerSGDState

    shapes = [(700, 1100), (1100,), (256, 512)]
    st = PowerSGDState(shapes, 2, matrix_approximation_rank=4, start_powerSGD_iter=0, device=DEV)
    g = [torch.from_numpy(x).to(DEV) for x in grads_for(shapes, 2, 0)]
    names = st.profile_kind_names()
    assert "pass1" in names and "pass3" in names
    st.step(g)
    torch.cuda.synchronize()
    st.profile_select(["pass1"])
    for _ in range(3):
        st.step(g)
    rec = st.profile_read()
    assert rec["pass1"][0] == 3 and rec["pass1"][1] > 0.0
    assert all(v[0] == 0 for k, v in rec.items() if k != "pass1")
    st.profile(True)
    st.step(g)
    rec = st.profile_read()
    assert rec["pass1"][0] == 1 and rec["pass2"][0] == 1 and rec["pass3"][0] == 1
    st.profile(False)
    assert not st.status()
    st.close()


@pytest.mark.parametrize("rank", [4, 16])
def test_bounded_wait_timeout_leaves_state_unchanged(rank):
    """A grid barrier of the cooperative Gram-Schmidt stage that can never
    complete (it waits for one arrival more than the launch has CTAs): every
    CTA gives up after its bounded polls, the step reports PSGD_ETIMEOUT and
    is not committed, the GPU stays usable, and the next steps equal, bit for
    bit, those of a state that never saw the failed step (at rank 16 the
    tensor-core operand images are rebuilt from the committed factors)."""
    import ctypes

    from powersgd_rank_gradient_gb300 import PowerSGDState, _lib

    world = 2
    make = lambda: PowerSGDState(ALIGNED, world, matrix_approximation_rank=rank, start_powerSGD_iter=0,
                                 min_compression_rate=0.25, device=DEV)
    a, b = make(), make()
    dev = lambda k: [torch.from_numpy(x).to(DEV) for x in grads_for(ALIGNED, world, k)]
    for st in (a, b):
        st.step(dev(0))
        assert not st.status()
    nt = [t for t in range(len(ALIGNED)) if len(ALIGNED[t]) > 1]
    snap = lambda st: ([st.get_q(t).clone() for t in nt], [st.get_p(t).clone() for t in nt],
                       [st.get_error(w).cpu().clone() for w in range(world)])
    before = snap(a)
    L = _lib.lib()
    L.psgd_internal_force_wait_timeout.argtypes = [ctypes.c_void_p]
    L.psgd_internal_force_wait_timeout.restype = ctypes.c_int
    assert L.psgd_internal_force_wait_timeout(a._h) == 0
    a.step(dev(1))
    with pytest.raises(_lib.PsgdError) as err:
        a.status()
    assert err.value.code == _lib.PSGD_ETIMEOUT
    after = snap(a)
    for xs, ys in zip(before, after):
        for x, y in zip(xs, ys):
            assert torch.equal(x, y)
    for k in (2, 3):
        oa, ob = a.step(dev(k)), b.step(dev(k))
        assert not a.status() and not b.status()
        assert torch.equal(oa, ob)
    for xs, ys in zip(snap(a), snap(b)):
        for x, y in zip(xs, ys):
            assert torch.equal(x, y)
    a.close()
    b.close()


@pytest.mark.parametrize("rank,world,which", [(4, 2, "mixed"), (4, 8, "mixed"), (3, 9, "mixed"),
                                              (16, 2, "aligned"), (32, 3, "aligned")])
def test_one_half_error_store_same_bits(rank, world, which):
    """psgd_set_error_store_halves(1): the error store kept once, pass 1
    writing M_w over the residual it has just read (chunk-stationary,
    tensor-core and element paths; the M-bar scratch at W >= 3) gives the same
    bits as the two-half store, every step, with one half less memory; the
    call is refused once a step was taken."""
    from powersgd_rank_gradient_gb300 import PowerSGDState, _lib

    shapes = MIXED if which == "mixed" else ALIGNED
    kw = dict(matrix_approximation_rank=rank, start_powerSGD_iter=0,
              min_compression_rate=1.0 if which == "mixed" else 0.25, device=DEV)
    one, two = PowerSGDState(shapes, world, **kw), PowerSGDState(shapes, world, **kw)
    before = one.workspace_bytes()
    one.set_error_store_halves(1)
    assert 0 < one.workspace_bytes() < before
    for k in range(3):
        g = [torch.from_numpy(x).to(DEV) for x in grads_for(shapes, world, k)]
        o1 = one.step(g).clone()
        o2 = two.step(g).clone()
        assert not one.status() and not two.status()
        assert torch.equal(o1, o2), k
    for w in range(world):
        assert torch.equal(one.get_error(w), two.get_error(w))
    with pytest.raises(_lib.PsgdError):
        one.set_error_store_halves(2)
    one.close()
    two.close()
