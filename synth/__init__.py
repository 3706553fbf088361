"""Seeded synthetic workloads for the layer-wise KV sparsification hot path.

This package holds shapes, per-layer budgets and seeded random draws only; it
holds none of the method's arithmetic.  Both the CPU oracle (under tests) and
the CUDA path consume the bytes it produces.
"""
from .workloads import (  # noqa: F401
    Workload,
    WORKLOADS,
    tiny,
    llama3_8b,
    continuous_batching,
    long_context,
    shared_prefix,
    bf16_bits,
    bf16_to_f64,
    bf16_to_f32,
    prefill_qkv,
    decode_qkv,
    sink_direction,
    shuffled_block_order,
    uniform_scores,
)
