"""Seeded synthetic workloads (inputs only; no FFN arithmetic)."""
from .workloads import (  # noqa: F401
    WORKLOADS,
    FFNSpec,
    bf16_bits_to_float32,
    make_dy,
    make_inputs,
    make_stack,
    make_weights,
    make_x,
    outlier_rows,
    random_bf16_matrix,
    round_to_bf16_bits,
    stack_layer_mean_active,
    stack_layer_spec,
)
