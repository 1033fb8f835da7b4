"""Seeded synthetic inputs for the routed-expert MoE layer iteration.

This package holds random draws, rounding to the storage dtype and commit
schedules only: none of the layer's arithmetic. Both the oracle-driven tests
and the GPU benchmark take their inputs from here, so the two sides see the
same values without sharing any code of the method itself.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_to_f64,
    block_masks,
    expert_payload,
    experts_payload,
    hidden_states,
    round_payload,
    router_payload,
    shared_experts_payload,
    shared_payload,
    sweep_workload,
    to_f64,
)
