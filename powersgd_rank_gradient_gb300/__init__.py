"""GB300-native PowerSGD communication-hook step (CUDA kernels behind a C ABI).

``PowerSGDState`` / ``powerSGD_hook`` load ``libpsgd.so`` (built in-tree by
``powersgd_rank_gradient_gb300.build``) on first use; nothing here falls back
to a CPU implementation.
"""


def __getattr__(name):
    if name in ("PowerSGDState", "powerSGD_hook", "BatchedPowerSGDState", "batched_powerSGD_hook",
                "PowerSGDGroup"):
        from . import hook

        return getattr(hook, name)
    if name in ("DataParallelPowerSGDState", "dp_powerSGD_hook"):
        from . import dp

        return getattr(dp, name)
    raise AttributeError(name)
