"""GB300-native NVFP4 weight-only (W4A16) sigmoid-top-k MoE decode layer.

The compute path is the CUDA library built from ``csrc/`` for sm_103a
(``build.build()``); this package only binds its C ABI (``moe``).
"""
from .moe import (EXPORTED, LIB_PATH, MOE_OK, MoEError, MoELayer, lib, last_error,  # noqa: F401
                  make_config, moe_check, moe_config, moe_debug_dequant, moe_decode_forward,
                  moe_decode_forward_host, moe_destroy, moe_get_info, moe_init, moe_layer_info,
                  moe_route_topk_static, moe_stage_down, moe_stage_gate_up, moe_trace_attach,
                  moe_stage_route, moe_debug_inject, moe_quant_fos, MOE_INJECT_WAIT_STALL,
                  moe_weights, to_device)
