"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

Holds only input construction (value streams and engine-side metadata); none
of the attention or cache-write arithmetic.
"""
from . import configs, data, gen  # noqa: F401
