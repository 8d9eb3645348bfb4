"""GB300-native fused residual-add + RMSNorm + block-scaled FP4 quantization.

The computation lives in libfp4q.so (hand-written sm_103a CUDA kernels behind
the C ABI in include/fp4q.h).  This package is a thin ctypes binding: the
functions named like the C entry points take raw device addresses, and
``add_rmsnorm_fp4quant`` / ``dequant`` marshal torch tensors (PyTorch provides
device memory and streams only).  There is no fallback: if the library is not
built, or a tensor is not on a CUDA device, the call raises.

Operation (FlashInfer page ``add_rmsnorm_fp4quant.py``, ``add_rmsnorm_fp4quant``):
residual <- input + residual; y = residual / sqrt(mean(residual^2) + eps) * weight;
y quantized to E2M1 with one scale per 16 (NVFP4, E4M3) or 32 (MXFP4, UE8M0)
elements, scales row-major and/or in the 128x4 tiled layout.

Around it: ``quantize_fp4`` (the same block quantization of x itself, FlashRT
``quantize_fp4_sfa_*``), and the consumer GEMM on the tensor cores,
``gemm_nvfp4_bf16`` / ``gemm_nvfp4_gelu`` (FlashRT ``nvfp4_gemm_*``: packed
E2M1 operands and their tiled scales in, bf16 or NVFP4 out, NVFP4 or MXFP4
operands, any K that is a multiple of 32), with ``fp4_gemm_variant`` and
``fp4_launch_shape`` reporting the launches the library would make.
Kernels that wait on asynchronous copies bound every wait; a call given a
device ``status`` word learns of a wait that ran out (``read_device_status``).
"""
from ._binding import (  # noqa: F401
    FP4_DT_BF16,
    FP4_DT_FP16,
    FP4_E4M3_B32,
    FP4_MXFP4,
    FP4_NVFP4,
    FP4_SF_BOTH,
    FP4_SF_ROWMAJOR,
    FP4_SF_SWIZZLED,
    FP4_OK,
    FP4_ERR_INVALID_ARG,
    FP4_ERR_UNSUPPORTED_SHAPE,
    FP4_ERR_MISALIGNED,
    FP4_ERR_CUDA,
    FP4_ERR_TIMEOUT,
    FP4_EPI_BF16,
    FP4_EPI_GELU_BF16,
    FP4_EPI_GELU_NVFP4,
    Fp4Error,
    add_rmsnorm_fp4quant,
    dequant,
    gemm_nvfp4_bf16,
    gemm_nvfp4_gelu,
    fp4_add_rmsnorm_quant,
    fp4_add_rmsnorm_quant_ex,
    fp4_add_rmsnorm_quant_gs,
    fp4_dequant,
    fp4_gemm_mxfp4_bf16,
    fp4_gemm_nvfp4_gelu_bf16,
    fp4_gemm_nvfp4_gelu_nvfp4,
    fp4_gemm_nvfp4_bf16,
    fp4_gemm_ex,
    fp4_read_device_status,
    read_device_status,
    fp4_quantize,
    fp4_last_cuda_error,
    fp4_launch_shape,
    fp4_gemm_variant,
    fp4_sf_size_bytes,
    fp4_status_string,
    debug_lib,
    fp4_debug_build,
    fp4_debug_configure,
    lib,
    lib_path,
    using_library,
    quantize_fp4,
)
