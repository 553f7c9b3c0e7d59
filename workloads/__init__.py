"""Seeded synthetic decode workloads shared by the tests, the oracle checks and
the benchmark.  Input data only: nothing here computes scores, selections or
attention."""
from .gen import CONFIGS, DecodeWorkload, RetopkWorkload, make_decode, make_retopk  # noqa: F401
