"""Seeded synthetic inputs (shared by the CUDA path's tests and the oracle; no MoE arithmetic)."""
from . import configs, gen  # noqa: F401
from .configs import WORKLOADS, Workload, scaled  # noqa: F401
