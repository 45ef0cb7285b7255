"""B300-native (sm_103a) forward of a Qwen3-style sparse Mixture-of-Experts block.

The compute runs in libmoe_b300.so (C ABI in include/moe_b300.h); this package
only marshals torch tensors into that ABI.  Build with
``python -m mixture_experts_layer_98_b300.build``.
"""
from .binding import (EXPORTS, LIB_PATH, MOE_PATH_AUTO, MOE_PATH_STREAMING,  # noqa: F401
                      MOE_PATH_TCGEN05, MOE_PATH_TCGEN05_DECODE, MOE_PATH_TCGEN05_PAIR,
                      MOE_PATH_WARP_MMA,
                      MOE_PATH_TCGEN05_WT, MoEError,
                      PackedExperts, Q4Experts, lib, moe_dequantize_experts_q4,
                      moe_forward_q4, moe_forward_host_q4, moe_q4_experts_bytes,
                      moe_quantize_experts_q4,
                      moe_dbg_combine, moe_dbg_permute, moe_dbg_wait_timeout, moe_forward_host_packed,
                      moe_forward_opts, moe_forward_packed, moe_pack_experts, moe_packed_experts_bytes,
                      moe_dbg_route_from_logits, moe_device_status, moe_forward,
                      moe_forward_host, moe_kernel_launch_count, moe_last_expert_counts,
                      moe_set_expert_path, moe_set_next_stage_events, moe_set_stage_timing,
                      moe_stage_times,
                      moe_workspace_bytes, STAGE_NAMES)

forward = moe_forward
