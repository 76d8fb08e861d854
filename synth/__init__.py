"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This package draws random tensors of the workload shapes and nothing else: it
holds none of the MoE layer's arithmetic.
"""
from .moe_inputs import (  # noqa: F401
    ATTN_CONFIGS,
    CONFIGS,
    AttnShape,
    LayerShape,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    make_attention,
    make_layer,
    make_output_grad,
    make_tokens,
)
