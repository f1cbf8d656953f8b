"""B300 (sm_103a) NVFP4 quantized linear layers.

Dynamic bfloat16 -> NVFP4 activation quantization, offline weight
quantization and a tcgen05 block-scaled FP4 GEMM with bfloat16 output, as a
C-ABI library of hand-written CUDA kernels (``include/nvfp4.h``,
``libnvfp4_b300.so``) with this thin PyTorch binding on top. The formats are
those of the "nvfp4-gemma4" and "nvfp4-difusion" pages (section 2 of each).
"""
from .ops import (  # noqa: F401
    SF_ROW_MAJOR,
    SF_MMA_128x4,
    LINEAR_UNFUSED,
    LINEAR_FUSED,
    SCALE_ABSMAX,
    SCALE_FOUR_OVER_SIX,
    SCALE_MSE,
    NVFP4Error,
    sf_bytes,
    sf_shape,
    nvfp4_global_scale,
    nvfp4_quantize,
    nvfp4_quantize_weight,
    nvfp4_sf_to_mma_layout,
    nvfp4_gemm,
    nvfp4_linear,
    nvfp4_linear_noalloc,
    nvfp4_linear_bias_requant,
    nvfp4_linear_bias_requant_dynamic,
    nvfp4_linear_grouped,
    nvfp4_linear_lora,
    pack_weight_groups,
    gemm_workspace_bytes,
    linear_workspace_bytes,
    nvfp4_device_error,
    nvfp4_debug_set_fault_injection,
)
from ._native import LIB_PATH, load as load_library  # noqa: F401
