"""causal_scaled_dot_gb300 -- causal scaled dot-product attention forward on GB300.

The compute lives in ``libattn.so`` (hand-written CUDA for sm_103a behind the C
ABI declared in ``include/attn.h``).  This package builds and loads that
library and marshals arguments into it; see ``native.py``.
"""
from .workloads import WORKLOADS, BY_NAME, HEADLINE, SMALL, Workload  # noqa: F401

__all__ = ["WORKLOADS", "BY_NAME", "HEADLINE", "SMALL", "Workload"]
