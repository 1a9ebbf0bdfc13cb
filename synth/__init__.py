"""Seeded synthetic workloads (random draws only, no CompKV arithmetic)."""
from .workloads import *  # noqa: F401,F403
from .workloads import WORKLOADS, Workload, capacity_tokens, queries, sequence_lengths, \
    sequence_tokens, step_queries, small_variant  # noqa: F401
