"""Seeded synthetic inputs for the fused MoE expert computation.

This module is shared by the tests, the smoke check and the benchmark.  It
draws hidden states, router logits, expert maps and already-quantised weights
(codes + scales, the form a checkpoint ships them in).  It holds none of the
expert computation itself: no sort, no GEMM, no activation, no activation
quantiser.  Weight codes for the formats whose recipe starts from a float
weight (FP8, NVFP4) are made with torch library casts (float8_e4m3fn) and a
nearest-value lookup -- checkpoint synthesis, done once, outside the timed
region; the oracle and the CUDA path each decode those codes on their own.

See ``gen.py`` for the per-workload recipes.
"""
from .gen import (WORKLOADS, Workload, make_custom, make_workload, to_host, workload_names)

__all__ = ["WORKLOADS", "Workload", "make_custom", "make_workload", "to_host", "workload_names"]
