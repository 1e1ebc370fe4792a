"""Seeded synthetic inputs for the KV-compression hot path.

This package only synthesises inputs (caches, probes, slot boundaries, hidden
states, decode-step vectors).  It holds none of the compression method's
arithmetic, and both the CPU oracle's tests and the GPU path's tests draw their
inputs from here.
"""
from .workloads import (  # noqa: F401
    CONFIGS,
    Workload,
    SeqInputs,
    decode_inputs,
    get_config,
    hidden_states,
    make_workload,
    round_bf16,
    small_config,
)
