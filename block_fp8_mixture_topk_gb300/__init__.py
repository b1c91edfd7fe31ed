"""GB300-native block-FP8 fused MoE expert layer.

Thin Python binding over the C ABI in ``include/moefp8.h`` (``libmoefp8.so``,
built in-tree for sm_103a).  PyTorch provides device memory and streams only;
every step of the layer runs in the library's CUDA kernels.  If the library is
missing or cannot be built, the functions raise: there is no CPU fallback.
"""
from .ops import (  # noqa: F401
    MOE_BLOCK_M,
    MoeError,
    RoutingParams,
    fp8_block_grouped_gemm,
    fp8_block_quant_weight,
    fp8_group_quant,
    library_path,
    moe_align_permute,
    moe_combine_pairs,
    moe_device_supported,
    moe_fp8_block_forward,
    moe_fp8_block_forward_masked,
    moe_fp8_block_masked_workspace_size,
    moe_fp8_block_forward_kernel_count,
    moe_fp8_block_decode_path,
    moe_fp8_block_pair_path,
    moe_fp8_block_pack_scales,
    moe_fp8_block_pack_weights,
    moe_fp8_block_workspace_size,
    moe_get_device_status,
    moe_max_padded_rows,
    moe_max_tiles,
    moe_mxfp8_pack_scales,
    moe_mxfp8_packed_scale_bytes,
    moe_mxfp8_quant_weight,
    moe_nvfp4_forward,
    moe_nvfp4_pack_weights,
    moe_nvfp4_packed_bytes,
    moe_nvfp4_quant_weight,
    moe_packed_scale_bytes,
    moe_route_topk,
    moe_selftest_bounded_wait,
    moe_unpermute_sum,
)
