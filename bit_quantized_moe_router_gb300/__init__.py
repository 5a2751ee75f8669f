"""GB300 (sm_103a) Q2_K mixture-of-experts FFN layer.

The layer runs in hand-written CUDA kernels behind the C ABI of
include/qs_moe.h (libqs_moe.so); `qs_moe` is its Python binding.
"""
from . import build
from . import qs_moe
from .qs_moe import (QS_BF16, QS_F32, QsError, alloc_workspace, make_experts, make_shape, make_shared,
                     qs_group_tokens, qs_moe_ffn, qs_moe_workspace_bytes, qs_q2k_down_combine,
                     qs_q2k_gemv_grouped, qs_q2k_quantize, qs_read_device_status, qs_route_topk,
                     qs_shared_expert_ffn, qs_workspace_init)

__all__ = ["build", "qs_moe", "QS_BF16", "QS_F32", "QsError", "alloc_workspace", "make_experts", "make_shape",
           "make_shared", "qs_group_tokens", "qs_moe_ffn", "qs_moe_workspace_bytes", "qs_q2k_down_combine",
           "qs_q2k_gemv_grouped", "qs_q2k_quantize", "qs_read_device_status", "qs_route_topk",
           "qs_shared_expert_ffn", "qs_workspace_init"]
