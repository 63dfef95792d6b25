"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the bench.

This package only draws random numbers and arranges them into the tensors a
routed-MoE forward consumes (token activations, router weights, expert
weights, an optional per-expert router bias, an optional shared expert's
weights).  It holds none of the method's
arithmetic: no quantization, routing, permutation or GEMM lives here, so both
the CPU oracle and the CUDA path can take their inputs from it without sharing
any computation.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    MoEShape,
    Workload,
    make_activations,
    make_router,
    make_shared_weights,
    make_weights,
    make_workload,
    zipf_router_bias,
)
