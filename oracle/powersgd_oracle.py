"""fp64 CPU oracle for the PowerSGD communication-hook step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
product path (the CUDA library and its Python binding) never calls it, and it
shares no code with that path: no kernels, no helpers, no constants.

What it computes, and where each step comes from:

* "DDP Communication Hooks" (PyTorch 1.11 docs), section "PowerSGD State":
  ``PowerSGDState(process_group, matrix_approximation_rank=1,
  start_powerSGD_iter=1000, min_compression_rate=2, use_error_feedback=True,
  warm_start=True, orthogonalization_epsilon=0, random_seed=0, ...)``;
  item 3 gives the compression gate
  ``(num_rows + num_cols) * matrix_approximation_rank * min_compression_rate
  < num_rows * num_cols``; item 4 gives the epsilon of the orthogonalisation.
* same page, section "PowerSGD Hooks", ``powerSGD_hook`` steps 1 to 3.7
  (split, uncompressed allreduce, P = MQ, allreduce P, orthogonalise P,
  Q = M^T P, allreduce Q, M ~ P Q^T), plus the note that vanilla allreduce runs
  for the first ``start_powerSGD_iter`` iterations and the warning that error
  feedback needs memory the size of the gradients.
* same page, "Default Communication Hooks", ``allreduce_hook``: the allreduce
  result is the MEAN over workers.
* "DDP Communication Hooks" (spec-zone.ru translation of a later version),
  "PowerSGD State" item 5: ``batch_tensors_with_same_shape`` only changes how
  same-shape tensors are scheduled, not the values.
* "Automatic Mixed Precision package - torch.cuda.amp", ``GradScaler``:
  gradients are unscaled (divided by the scale) and checked for inf/NaN; a
  step that sees one is skipped and leaves the parameters (here: the hook's
  state) untouched.

Readings taken where the pages are silent:
epsilon is added to the column NORM in the denominator; "allreduce" is the mean
over the W simulated replicas; each replica computes its own P = M_w Q and the
P's are then averaged (no linearity shortcut here); the initial Q is a standard
normal draw that is orthogonalised, while a warm-started Q is used as is; the
error buffer starts at zero and is kept per replica; tensors of fewer than two
dimensions are never compressed; a >=2-D tensor is viewed as
(shape[0], prod(shape[1:])); the effective rank is min(r, rows, cols).

Everything is float64 NumPy, written for a reader to check against the pages,
not for speed.  Random draws are INPUTS: the caller injects the standard-normal
sample for Q with ``set_q_draw``.  If none was injected the oracle draws one
from ``numpy.random.default_rng((random_seed, tensor, draw))``; that stream is
not meant to match any other implementation.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SKIPPED = "skipped"
OK = "ok"


@dataclass
class TensorPlan:
    """One per-parameter tensor of the flat bucket.

    "PowerSGD Hooks", powerSGD_hook step 1: the flat 1-D bucket is viewed as
    a list of per-parameter tensors and split into a compressed group and an
    uncompressed group (which holds every vector tensor).
    """

    index: int
    shape: tuple
    offset: int          # first element of the tensor in the flat bucket
    numel: int
    compressed: bool
    rows: int = 0        # shape[0]
    cols: int = 0        # prod(shape[1:])
    rank: int = 0        # min(matrix_approximation_rank, rows, cols)


def plan_bucket(shapes, matrix_approximation_rank, min_compression_rate):
    """Split a bucket into per-parameter tensors and apply the gate.

    "PowerSGD State" item 3: a tensor is compressed only if
    (num_rows + num_cols) * matrix_approximation_rank * min_compression_rate
    < num_rows * num_cols (strict).  "PowerSGD Hooks" step 1.2: all vector
    tensors (biases) go uncompressed.
    """
    plans = []
    offset = 0
    for index, shape in enumerate(shapes):
        shape = tuple(int(d) for d in shape)
        numel = 1
        for d in shape:
            numel *= d
        if len(shape) < 2:
            plans.append(TensorPlan(index, shape, offset, numel, False))
        else:
            rows = shape[0]
            cols = numel // rows if rows > 0 else 0
            # Python compares the float left side with the int right side exactly.
            lhs = (rows + cols) * matrix_approximation_rank * float(min_compression_rate)
            compressed = rows > 0 and cols > 0 and lhs < rows * cols
            rank = min(matrix_approximation_rank, rows, cols) if compressed else 0
            plans.append(TensorPlan(index, shape, offset, numel, compressed, rows, cols, rank))
        offset += numel
    return plans


def allreduce_mean(arrays):
    """The allreduce of the simulated job: the mean over the replicas
    ("Default Communication Hooks", allreduce_hook: the aggregated tensor is
    divided by the number of workers, i.e. the mean)."""
    acc = np.zeros_like(np.asarray(arrays[0], dtype=np.float64))
    for a in arrays:
        acc = acc + a
    return acc / len(arrays)


def compute_p(m, q):
    """Step 3.2: P = M Q (one replica)."""
    return m @ q


def compute_q(m, p):
    """Step 3.5: Q = M^T P (one replica)."""
    return m.T @ p


def decompress(p, q):
    """Step 3.7: M is approximated by P Q^T."""
    return p @ q.T


def orthogonalize(matrix, epsilon):
    """Gram-Schmidt over the columns, in column order.

    "PowerSGD Hooks" step 3.4 ("Orthogonalizes each P") and "PowerSGD State"
    item 4: epsilon is added so that an all-zero column does not divide by
    zero.  Reading: column i is divided by (||column i|| + epsilon), then its
    projection is removed from every later column.  With epsilon = 0 an
    all-zero column gives NaN, as the pages warn.
    """
    a = np.array(matrix, dtype=np.float64, copy=True)
    rank = a.shape[1]
    with np.errstate(divide="ignore", invalid="ignore"):
        for i in range(rank):
            norm = math.sqrt(float(np.dot(a[:, i], a[:, i])))
            a[:, i] = a[:, i] / (norm + epsilon)
            for j in range(i + 1, rank):
                a[:, j] = a[:, j] - np.dot(a[:, i], a[:, j]) * a[:, i]
    return a


@dataclass
class PowerSGDOracle:
    """Hyper-parameters and per-tensor state ("PowerSGD State").

    The simulated data-parallel job has ``world_size`` replicas; each replica
    w hands the hook its own flat gradient bucket g_w.
    """

    shapes: list
    world_size: int
    matrix_approximation_rank: int = 1
    start_powerSGD_iter: int = 1000
    min_compression_rate: float = 2.0
    use_error_feedback: bool = True
    warm_start: bool = True
    orthogonalization_epsilon: float = 0.0
    random_seed: int = 0
    batch_tensors_with_same_shape: bool = False
    iter: int = 0
    plans: list = field(default_factory=list)
    q: dict = field(default_factory=dict)          # tensor -> Q (cols x rank), float64
    error: dict = field(default_factory=dict)      # (replica, tensor) -> E (rows x cols)
    last_p: dict = field(default_factory=dict)     # tensor -> orthogonalised P of the last step
    _draws: dict = field(default_factory=dict)     # tensor -> injected N(0,1) sample
    _draw_count: dict = field(default_factory=dict)

    def __post_init__(self):
        self.plans = plan_bucket(self.shapes, self.matrix_approximation_rank,
                                 self.min_compression_rate)
        self.numel = sum(p.numel for p in self.plans)

    # -- inputs ------------------------------------------------------------
    def set_q_draw(self, tensor, draw):
        """Inject the standard-normal sample used the next time tensor ``tensor``
        needs a fresh Q ("PowerSGD Hooks" step 3.1: Q is initialised from a
        standard normal distribution and orthogonalised)."""
        plan = self.plans[tensor]
        draw = np.asarray(draw, dtype=np.float64).reshape(plan.cols, plan.rank)
        self._draws[tensor] = draw.copy()

    def set_warm_q(self, tensor, q):
        """Install a warm-start Q as is (no orthogonalisation)."""
        plan = self.plans[tensor]
        self.q[tensor] = np.asarray(q, dtype=np.float64).reshape(plan.cols, plan.rank).copy()

    def _fresh_draw(self, tensor):
        if tensor in self._draws:
            return self._draws.pop(tensor)
        plan = self.plans[tensor]
        count = self._draw_count.get(tensor, 0)
        self._draw_count[tensor] = count + 1
        rng = np.random.default_rng((self.random_seed, tensor, count))
        return rng.standard_normal((plan.cols, plan.rank))

    # -- the hook ----------------------------------------------------------
    def step(self, grads, inv_loss_scale=1.0):
        """One call of the hook on the W replicas' buckets.

        Returns ``(status, out)``: ``out`` is the float64 flat bucket every
        replica receives (None when the step is skipped).
        """
        assert len(grads) == self.world_size
        g = []
        for w in range(self.world_size):
            flat = np.asarray(grads[w]).reshape(-1)
            assert flat.size == self.numel
            # GradScaler unscale: divide by the scale (multiply by its inverse).
            g.append(flat.astype(np.float64) * float(inv_loss_scale))

        # GradScaler: a step whose gradients hold inf/NaN is skipped and leaves
        # the state as it was.  The iteration counter still advances (the hook
        # counts its own calls).
        if not all(np.all(np.isfinite(x)) for x in g):
            self.iter += 1
            return SKIPPED, None

        out = np.zeros(self.numel, dtype=np.float64)

        # "Note that this communication hook enforces vanilla allreduce for the
        # first state.start_powerSGD_iter iterations."
        if self.iter < self.start_powerSGD_iter:
            out = allreduce_mean(g)
            self.iter += 1
            return OK, out

        # Step 2: the uncompressed tensors are allreduced (mean) without
        # compression and copied back; no error feedback on this path.
        for plan in self.plans:
            if plan.compressed:
                continue
            sl = slice(plan.offset, plan.offset + plan.numel)
            out[sl] = allreduce_mean([g[w][sl] for w in range(self.world_size)])

        # Step 3, tensor by tensor.  ``batch_tensors_with_same_shape`` changes
        # only how the real hook groups its matmuls, so the values here do not
        # depend on it.
        for plan in self.plans:
            if not plan.compressed:
                continue
            t = plan.index
            sl = slice(plan.offset, plan.offset + plan.numel)
            m_w = []
            for w in range(self.world_size):
                mat = g[w][sl].reshape(plan.rows, plan.cols).copy()
                if self.use_error_feedback and (w, t) in self.error:
                    mat = mat + self.error[(w, t)]
                m_w.append(mat)

            # 3.1: a fresh Q (standard normal, orthogonalised) unless a warm Q
            # from the previous step exists and warm_start is on.
            if self.warm_start and t in self.q:
                q = self.q[t]
            else:
                q = orthogonalize(self._fresh_draw(t), self.orthogonalization_epsilon)

            # 3.2 + 3.3: each replica computes P = M Q, then the Ps are averaged.
            p = allreduce_mean([compute_p(m_w[w], q) for w in range(self.world_size)])

            # 3.4: orthogonalise P.
            p = orthogonalize(p, self.orthogonalization_epsilon)

            # 3.5 + 3.6: each replica computes Q = M^T P, then the Qs are averaged.
            q_new = allreduce_mean([compute_q(m_w[w], p) for w in range(self.world_size)])

            # 3.7: the decompressed tensor P Q^T replaces the gradient.
            m_hat = decompress(p, q_new)
            out[sl] = m_hat.reshape(-1)

            # Error feedback: each replica keeps what the compression lost.
            if self.use_error_feedback:
                for w in range(self.world_size):
                    self.error[(w, t)] = m_w[w] - m_hat

            self.q[t] = q_new
            self.last_p[t] = p

        self.iter += 1
        return OK, out

    # -- views for tests -----------------------------------------------------
    def error_of(self, replica, tensor):
        plan = self.plans[tensor]
        return self.error.get((replica, tensor), np.zeros((plan.rows, plan.cols)))

    def compression_stats(self):
        """Element counts before and after compression ("PowerSGD State":
        compression statistics are logged every
        compression_stats_logging_frequency iterations)."""
        before = sum(p.numel for p in self.plans)
        after = sum((p.rows + p.cols) * p.rank if p.compressed else p.numel
                    for p in self.plans)
        return before, after


@dataclass
class BatchedPowerSGDOracle:
    """batched_powerSGD_hook ("PowerSGD Hooks", batched_powerSGD_hook steps
    1-9): the whole flat bucket of N elements is viewed as one square matrix
    of side ceil(sqrt(N)) with zero padding, compressed by one PowerSGD step,
    and the result truncated to N elements.  Reading: error feedback (one
    residual per replica) covers the whole padded square, as the per-tensor
    hook's covers each compressed tensor; there is no compression-rate gate.
    """

    numel: int
    world_size: int
    matrix_approximation_rank: int = 1
    start_powerSGD_iter: int = 1000
    use_error_feedback: bool = True
    warm_start: bool = True
    orthogonalization_epsilon: float = 0.0
    random_seed: int = 0
    iter: int = 0
    q: object = None
    error: dict = field(default_factory=dict)
    last_p: object = None
    _draw: object = None

    def __post_init__(self):
        self.side = math.isqrt(self.numel - 1) + 1 if self.numel > 0 else 0
        self.rank = min(self.matrix_approximation_rank, self.side)

    def set_q_draw(self, draw):
        self._draw = np.asarray(draw, dtype=np.float64).reshape(self.side, self.rank).copy()

    def step(self, grads, inv_loss_scale=1.0):
        g = [np.asarray(x).reshape(-1).astype(np.float64) * float(inv_loss_scale) for x in grads]
        assert len(g) == self.world_size and all(x.size == self.numel for x in g)
        if not all(np.all(np.isfinite(x)) for x in g):
            self.iter += 1
            return SKIPPED, None
        if self.iter < self.start_powerSGD_iter:
            self.iter += 1
            return OK, allreduce_mean(g)
        n = self.side
        # 1: the square view with zero padding (plus the replica's residual)
        m_w = []
        for w in range(self.world_size):
            sq = np.zeros(n * n)
            sq[:self.numel] = g[w]
            sq = sq.reshape(n, n)
            if self.use_error_feedback and w in self.error:
                sq = sq + self.error[w]
            m_w.append(sq)
        # 2: Q from a standard-normal draw, orthogonalised, unless warm
        if self.warm_start and self.q is not None:
            q = self.q
        else:
            if self._draw is None:
                rng = np.random.default_rng((self.random_seed, self.iter))
                self._draw = rng.standard_normal((n, self.rank))
            q = orthogonalize(self._draw, self.orthogonalization_epsilon)
            self._draw = None
        # 3-5: P = M Q, allreduce (mean), orthogonalise
        p = orthogonalize(allreduce_mean([compute_p(m, q) for m in m_w]), self.orthogonalization_epsilon)
        # 6-7: Q = M^T P, allreduce (mean)
        q_new = allreduce_mean([compute_q(m, p) for m in m_w])
        # 8: M ~ P Q^T; 9: truncate to the original length
        m_hat = decompress(p, q_new)
        if self.use_error_feedback:
            for w in range(self.world_size):
                self.error[w] = m_w[w] - m_hat
        self.q = q_new
        self.last_p = p
        self.iter += 1
        return OK, m_hat.reshape(-1)[:self.numel].copy()

    def error_of(self, replica):
        return self.error.get(replica, np.zeros((self.side, self.side)))
