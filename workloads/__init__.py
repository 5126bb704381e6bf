"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle-side checks."""
from .synth import MODES, WORKLOADS, Workload, make_inputs, routing, scaled, to_numpy  # noqa: F401
