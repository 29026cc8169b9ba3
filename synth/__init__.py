"""Seeded synthetic inputs for tree-verification workloads (input generation only)."""

from .gen import (  # noqa: F401
    WORKLOADS,
    Workload,
    Inputs,
    make_inputs,
    make_tree,
    logical_kv,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    eagle2_expand_step,
    build_eagle2_tree,
    binary_tree_parent,
    chain_parent,
)
