"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package holds input generation only (Qwen3-shaped caches, calibration
queries, block tables); it contains none of the compression method's arithmetic.
"""
from .generate import (  # noqa: F401
    Workload,
    WORKLOADS,
    generate,
    generate_layer,
    unit_rows,
    seed_for,
    sequence_samples,
    vonmises,
)
