"""GB300-native hot path of one Colibri GLM-5.2 MoE layer.

Route (sigmoid top-k) -> Union (group pairs by expert) -> int4 SwiGLU expert FFN
(routed + shared) -> score-weighted combine -> Learn (hit counters), as the C ABI
of ``include/moe.h`` over hand-written sm_103a kernels.  This package is the
thin Python binding of that library (argument marshalling only).
"""
from . import _binding  # noqa: F401
from ._binding import (  # noqa: F401
    MOE_DEVERR_BAD_EXPERT, MOE_DEVERR_BOUNDS, MOE_DEVERR_SCALE_RANGE, MOE_DEVERR_TIMEOUT, MOE_ERR_CUDA, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED,
    MOE_ERR_WORKSPACE, MOE_MODE_AUTO, MOE_MODE_DECODE, MOE_MODE_HYBRID, MOE_MODE_PREFILL, MOE_OK, LayerWeights, MoeError,
    device_error, expert_q_bytes, expert_s_count, ffn_workspace_bytes, header_functions, layer_workspace_bytes,
    lib, moe_combine, moe_expert_ffn_int4, moe_expert_ffn_int4_noalloc, moe_hits, moe_layer_forward, moe_rms_norm,
    moe_route, moe_union, status_str, workspace, ExpertTier, tier_workspace_bytes, moe_layer_forward_tier,
    MOE_ERR_STALE, usage_save, usage_load, usage_top, moe_layer_forward_host, layer_host_workspace_bytes,
    moe_layer_forward_norm,
)
