"""Seeded synthetic inputs shared by the CUDA library's tests/benchmark and the CPU oracle."""
from .workloads import WORKLOADS, Workload, get, micro, make_x, make_routing, make_weights, make_all, active_experts  # noqa: F401
