"""Seeded synthetic inputs for the fused FP4-weight MoE layer.

This package is shared by the tests, the benchmark and the oracle harness. It
draws random numbers and writes synthetic checkpoints; it contains none of the
layer's arithmetic (no dequantisation, no GEMV/GEMM, no activation, no
router-weighted sum).

The pages measure on model checkpoints (DS4-Flash, Kimi, DeepSeek, GLM, Qwen
layers) that are not available here; the seeded draws below stand in for them
with the pages' expert geometries.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    Workload,
    draw_activations,
    draw_routing,
    draw_routing_pool,
    encode_mxfp4,
    encode_nvfp4,
    make_workload,
    make_expert_weights,
)
