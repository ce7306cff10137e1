"""Seeded synthetic inputs for the MXFP4 routed-MoE layer.

This package only draws random numbers and arranges them in the storage
layout the layer consumes. It holds none of the layer's arithmetic, so both
the CPU oracle and the CUDA path can take their inputs from it.
"""

from .moe_inputs import (  # noqa: F401
    CONFIGS,
    interleave_gate_up,
    LayerSpec,
    make_layer,
    make_tokens,
    make_layer_torch,
    spec_for,
)
