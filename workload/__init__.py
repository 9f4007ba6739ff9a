"""Seeded synthetic workloads (shapes, seeds, counter-based input streams).

Shared by the oracle side and the CUDA side as an input source only; holds none of
the drafter's arithmetic.
"""
from .configs import ALL, BY_NAME, Workload, small_bf16  # noqa: F401
