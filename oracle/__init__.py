"""CPU oracle for fused residual-add + RMSNorm + block-scaled FP4 quantization.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
statement of what the CUDA library computes.  Only the tests, the smoke check
and the benchmark's CPU-baseline / reference leg may import it; the library in
``rmsnorm_fp4_quant_gb300`` never does, and the two share no code, tables or
helpers.  Inputs come from ``workloads`` (random numbers only).

Sources (web pages; section names as they appear there):
  * FlashInfer ``cute_dsl/add_rmsnorm_fp4quant.py`` (module docstring,
    ``AddRMSNormFP4QuantKernel.kernel`` phases 1-3, ``add_rmsnorm_fp4quant``
    Parameters / Returns / Notes) - the operation itself;
  * vLLM ``fused_wo_a`` (``FusedWoAKernel`` scale write-out) - the 128x4 scale
    tile order and zero-filled padding;
  * FlashRT ``fp4-gemm`` README (Tensor Contract, Available Functions,
    Validation) - the packed FP4 and SFA contract, validation by
    dequantisation, and the consumer GEMM (``oracle.gemm``).

Arithmetic is fp32 with every step correctly rounded (numpy float32 ops are
IEEE-754 round-to-nearest-even); the sum of squares is accumulated in fp64.
Where the pages leave a step open the reading taken is stated at the function.

Pinned by tests/test_oracle_*.py.  Parity unpinned: the nibble order inside a
byte and the sign of a zero code are conventions with no external pin.
"""
from .formats import (  # noqa: F401
    E2M1_GRID,
    bf16_round,
    fp16_round,
    round_to_dtype,
    e2m1_index_rne,
    e2m1_encode,
    e2m1_decode,
    e4m3_decode,
    e4m3_encode_rne,
    ue8m0_encode_ceil,
    ue8m0_decode,
)
from .add_rmsnorm_quant import (  # noqa: F401
    OracleResult,
    add_rmsnorm_fp4_quant,
    quantize,
    e4m3_scaled,
    swizzled_sf_offset,
    sf_size_bytes,
    dequant,
    block_size,
)
from .gemm import GemmResult, gelu, gemm_bf16, gemm_gelu_nvfp4  # noqa: F401
