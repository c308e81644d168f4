"""Seeded synthetic inputs for the NVFP4 W4A16 MoE decode layer.

This package draws random layers and activations in the canonical layout.  It
holds none of the layer's arithmetic (no decoding, routing, GEMV or combine):
both the CUDA path and the CPU oracle consume what it produces, and it imports
neither of them.
"""
from .synth import (BASE_SEED, CONFIGS, canonical_shapes, config, make_experts,  # noqa: F401
                    make_layer, make_layer_torch, make_router, make_x, make_x_token,
                    make_x_torch, selected_bytes)
