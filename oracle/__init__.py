"""fp64 CPU oracle (test infrastructure only; never imported by the product path)."""

from .powersgd_oracle import (  # noqa: F401
    OK,
    SKIPPED,
    BatchedPowerSGDOracle,
    PowerSGDOracle,
    TensorPlan,
    allreduce_mean,
    compute_p,
    compute_q,
    decompress,
    orthogonalize,
    plan_bucket,
)
