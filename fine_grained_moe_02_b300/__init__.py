"""Latent-routed top-k SwiGLU MoE layer forward on B300 (sm_103a).

The compute lives in libmoe.so (C ABI, include/moe.h); this package holds its
CUDA sources (csrc/), the build script and a thin ctypes binding.
"""
from .binding import (  # noqa: F401
    MoeError, MoeLayer, alloc_workspace, header_functions, lib, moe_check_dims, moe_clear_device_status,
    moe_combine, moe_dims, moe_forward_headlocal, moe_prepare_weights_headlocal,
    moe_workspace_size_headlocal, moe_ext, moe_forward_ext, moe_route_ext, moe_workspace_size_ext, moe_dispatch, moe_dispatch_indices, moe_dispatch_noalloc, moe_expert_ffn, moe_expert_gemm1,
    moe_expert_gemm1_gather, moe_expert_gemm2, moe_expert_gemm2_gated, moe_combine_rows, moe_forward_fused, moe_forward_folded, moe_prepare_router, moe_route_folded, moe_route_fused, moe_route_two_stage, moe_forward, moe_forward_host,
    moe_get_device_status, moe_prepare_weights, moe_route, moe_scratch_size, moe_selftest_timeout,
    moe_selftest_timeout_fused, moe_workspace_size,
    moe_workspace_size_host, status_string,
)
