"""Seeded synthetic workloads for the bit-plane KV scan.

This package only draws inputs (keys, values, queries, channel variances,
budgets, planted needles) and describes workload shapes and byte counts.
It holds none of the method's arithmetic, so both the CUDA path and the
CPU oracle can be fed from it without sharing any code with each other.
"""
from .gen import LayerInputs, gen_layer, unit_sigma  # noqa: F401
from .configs import CONFIGS, WorkloadConfig  # noqa: F401
