"""Seeded synthetic decode workloads (inputs only; no method arithmetic)."""
from .generators import (  # noqa: F401
    SEED_BASE,
    WORKLOADS,
    Workload,
    layer_seed,
    make_hyperplanes,
    make_layer,
    small_workload,
)
