"""GB300 (sm_103a) fused Mixture-of-Experts expert computation.

route -> gate/up grouped GEMM -> activation (SiLU / GELU / SwiGLU-OAI) ->
down grouped GEMM -> top-k weighted reduce, for bf16, FP8 (per-tensor,
per-channel, 128x128 block), MXFP4 and NVFP4 weights, behind the C ABI in
include/moe_experts.h (libmoe_gb300.so).  The Python names mirror the C entry
points; torch provides device memory and streams only.
"""
from ._binding import (ACT, AFMT, BLOCK_M, EXPORTS, GATE, LIB_PATH, WFMT, FusedExperts, MoEError,
                       Problem, Weight, lib, make_problem, make_weight, moe_abi_version,
                       moe_align_block_size, moe_align_block_size_scratch,
                       moe_align_capacity, moe_align_scratch_bytes, moe_fused_experts,
                       moe_fused_experts_noalloc, moe_noalloc_scratch_bytes,
                       moe_packed_weight_bytes, moe_prepare_weights,
                       moe_stage_timing, moe_stage_times, STAGES,
                       PATHS, moe_route_topk, SCORING, moe_mma_probe, MMA_KINDS,
                       moe_intermediate_size, moe_batched_workspace_size, moe_batched_experts,
                       moe_get_device_error, moe_grouped_gemm_w2_reduce,
                       moe_grouped_gemm_w13_act, moe_quant_act, moe_reset_device_error,
                       moe_selftest_bounded_wait, moe_w13_workspace_size, moe_workspace_size, stage2_format, status_str)

__all__ = [
    "ACT", "AFMT", "BLOCK_M", "EXPORTS", "GATE", "LIB_PATH", "WFMT", "FusedExperts", "MoEError",
    "Problem", "Weight", "lib", "make_problem", "make_weight", "moe_abi_version",
    "moe_align_block_size", "moe_align_block_size_scratch", "moe_align_capacity",
    "moe_align_scratch_bytes", "moe_fused_experts",
    "moe_fused_experts_noalloc", "moe_noalloc_scratch_bytes", "moe_packed_weight_bytes",
    "moe_prepare_weights", "moe_stage_timing", "moe_stage_times", "STAGES",
    "PATHS", "moe_route_topk", "SCORING", "moe_mma_probe", "MMA_KINDS",
    "moe_intermediate_size", "moe_batched_workspace_size", "moe_batched_experts",
    "moe_get_device_error",
    "moe_grouped_gemm_w2_reduce", "moe_grouped_gemm_w13_act", "moe_quant_act",
    "moe_reset_device_error", "moe_selftest_bounded_wait", "moe_w13_workspace_size", "moe_workspace_size", "stage2_format",
    "status_str",
]
