"""Seeded synthetic inputs for the LiLiCorr rerank path.

This package is the only code that both the CPU oracle and the CUDA path see.  It
draws random numbers and packs them into arrays; it performs none of the method's
arithmetic (no log-partition, no top-K, no network layer, no scoring).
"""
from .inputs import (  # noqa: F401
    CONFIGS,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_weights,
    make_workload,
    weight_shapes,
)
