"""Seeded synthetic inputs for paged-int8-KV prefill attention (shared by tests, bench and smoke).

This package only synthesises inputs (shapes, value distributions, page
placement); none of the attention arithmetic lives here.
"""
from .workloads import CONFIGS, Workload, Inputs, make_inputs, make_gate  # noqa: F401
