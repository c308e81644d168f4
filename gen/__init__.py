"""Seeded synthetic inputs for the NVFP4 W4A16 MoE decode layer.

This package draws random layers and activations in the canonical layout.  It
holds none of the layer's arithmetic (no decoding, routing, GEMV or combine):
both the CUDA path and the CPU oracle consume what it produces, and it imports
neither of them.
"""
from .synth import (CONFIGS, config, make_layer, make_router, make_experts,  # noqa: F401
                    make_x, make_x_token, canonical_shapes, selected_bytes)
