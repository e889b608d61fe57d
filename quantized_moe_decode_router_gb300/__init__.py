"""GB300-native quantized mixture-of-experts layer (sm_103a).

One MoE layer computed directly on block-quantized checkpoint weights
(NVFP4, MXFP4, int4/int8 group-64, FP8 block-128): router softmax + top-k,
expert dispatch, gate/up + SwiGLU, down projection and the weighted combine.
The compute runs in ``libqmoe.so`` (hand-written CUDA kernels behind the C ABI
of ``include/moe.h``); this package marshals arguments to it.
"""
from ._binding import (  # noqa: F401
    Layer, MoeError, QWeight, load, moe_check, moe_decode_forward, moe_decode_forward_timed, moe_dequantize,
    moe_experts_forward,
    moe_prefill_forward, moe_prefill_forward_timed,
    moe_quantize_act_mxfp4, moe_quantize_act_nvfp4, moe_route, decode_plan, status_string, workspace_init, workspace_layout, workspace_size,
    MOE_DECODE_MAX_TOKENS, MOE_FMT_FP8_B128, MOE_FMT_INT4_G64, MOE_FMT_INT8_G64, MOE_FMT_MXFP4, MOE_FMT_NONE,
    MOE_FMT_NVFP4,
)
from .device import DeviceLayer, to_device  # noqa: F401
