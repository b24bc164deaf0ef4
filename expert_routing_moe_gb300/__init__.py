"""GB300 (sm_103a) MoE routing layer: router + softmax/top-k, SERE batch
reroute, capacity dispatch, and a tcgen05 grouped SwiGLU FFN with the combine
fused in, behind the C ABI of include/moe_gb300.h."""
from ._abi import (MOE_DTYPE_BF16, MOE_DTYPE_F32, MOE_FFN_FUSE_COMBINE, MOE_FFN_ZERO_Y, MOE_OP_CALIBRATE,
                   MOE_OP_DISPATCH, MOE_OP_FFN, MOE_OP_ROUTE_DISPATCH, MOE_ROUTE_FROM_LOGITS, MOE_ROUTE_RENORM_TOPK, MoeError, SereParams, load,
                   moe_combine, moe_decode_layer, moe_dispatch_capacity, moe_residual_to_bf16, moe_ffn_grouped, moe_reroute_sere, moe_route, moe_route_dispatch,
                   moe_similarity_calibrate, moe_token_weights, status_string, workspace_size)
from .layer import MoELayer

__all__ = ["MoELayer", "SereParams", "MoeError", "load", "moe_route", "moe_route_dispatch", "moe_decode_layer", "moe_reroute_sere", "moe_dispatch_capacity",
           "moe_ffn_grouped", "moe_combine", "moe_residual_to_bf16", "moe_token_weights", "moe_similarity_calibrate", "workspace_size", "status_string",
           "MOE_DTYPE_BF16", "MOE_DTYPE_F32", "MOE_FFN_FUSE_COMBINE", "MOE_FFN_ZERO_Y", "MOE_OP_CALIBRATE", "MOE_OP_DISPATCH", "MOE_OP_FFN", "MOE_OP_ROUTE_DISPATCH", "MOE_ROUTE_FROM_LOGITS",
           "MOE_ROUTE_RENORM_TOPK"]
