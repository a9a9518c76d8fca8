"""MXFP8 (OCP MX, W8A8) block-scaled fused-MoE expert forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libmxmoe.so`` (hand-written CUDA,
tcgen05 tensor cores), with W4A8 (MXFP4 expert weights) and W4A4 (MXFP4
weights and expert inputs) variants and the dense MXFP8 / W4A4 linear (one
group of the grouped GEMM); ``api`` is
its thin Python binding and ``workloads``
the seeded synthetic inputs.  Importing ``api`` functions loads the library
lazily and raises if it has not been built.
"""

from .api import (  # noqa: F401
    MXFP8MoELayer, device_status, grouped_gemm_mxfp8, grouped_gemm_swiglu_quant_mxfp8,
    moe_finalize_routing, moe_forward_mxfp8, moe_forward_mxfp8_workspace_size,
    moe_forward_mxfp8_mma_scales, moe_route_permute_bf16, moe_route_quant_mxfp8, mx_quantize_3d,
    mx_scales_to_mma_layout, set_wait_limit_cycles, W4A8MoELayer, mx_quantize_fp4_3d,
    moe_forward_w4a8_mma_scales, MXFP8Linear, mxfp8_linear, mxfp8_linear_mma_scales,
    mxfp8_linear_workspace_size, set_gemm_2sm, set_gemm_chain, W4A4MoELayer, moe_forward_w4a4_mma_scales,
    MXFP4Linear, mxfp4_linear, mxfp4_linear_mma_scales, moe_router_gate_topk,
    mx_dequantize_bf16_2d, moe_forward_mxfp8_gated_mma_scales,
)
