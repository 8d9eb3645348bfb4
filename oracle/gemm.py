"""Oracle of the consumer GEMM: block-scaled FP4 A times FP4 B transposed, bf16 out.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the FlashRT ``fp4-gemm`` README:
  * Tensor Contract: ``a_packed`` uint8 (M, K/2), ``b_packed`` uint8 (N, K/2),
    ``sfa`` / ``sfb`` the 128x4 tiled scale buffers of (M, K) and (N, K),
    output bf16 (M, N);
  * Available Functions: ``nvfp4_gemm_bf16(..., alpha)``, the bias and residual
    epilogues ``nvfp4_gemm_bias_bf16``, ``nvfp4_gemm_residual_bf16``,
    ``nvfp4_gemm_bias_residual_bf16``;
  * Validation: the reference dequantises the very FP4 codes and scales the
    kernel reads and multiplies the dequantised matrices.

So, with deq() the exact E2M1-value-times-block-scale of ``oracle.dequant``:

    S[m, n]   = sum_k deq(A)[m, k] * deq(B)[n, k]          (fp64)
    out[m, n] = bf16( fp32( alpha * S[m, n] + bias[n] + residual[m, n] ) )

Readings where the README is silent:
  * the order of the epilogue terms: alpha scales the product only; bias
    (length N) and residual (M x N, bf16) are added after it, as the function
    names list them;
  * the sum is taken in fp64 (every product of two dequantised values is
    exact in fp64; the sum is exact up to fp64 rounding), then rounded once to
    fp32 and once to bf16 - the PyTorch-reference path of the Validation
    section (fp32 GEMM output cast to bf16).  A GPU accumulating in fp32 is
    compared against ``exact`` with the fp32 accumulation bound, not
    bit-for-bit;
  * ``bound`` = |alpha| * sum_k |deq(A)[m, k]| * |deq(B)[n, k]|, the scale of
    the rounding error of any summation order;
  * GELU (``nvfp4_gemm_bias_gelu_bf16`` / ``_nvfp4``; the README names it, the
    form is not given): the exact one, x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)),
    applied to alpha * S + bias;
  * the FP4-output epilogue (``nvfp4_gemm_bias_gelu_nvfp4`` "emits packed FP4
    plus CUTLASS SFA so the following projection can consume it"): the
    GELU values rounded once to fp32, then quantized by this oracle's
    producer rules (``oracle.quantize``, NVFP4, tiled scales), rows of the
    output as the rows of the next GEMM's A.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from .add_rmsnorm_quant import OracleResult, dequant, quantize
from .formats import bf16_round


@dataclasses.dataclass
class GemmResult:
    exact: np.ndarray     # (M, N) fp64: alpha * S + bias + residual
    out: np.ndarray       # (M, N) fp32 holding the bf16 result
    bound: np.ndarray     # (M, N) fp64: |alpha| * sum_k |a| |b|


def gelu(x) -> np.ndarray:
    """x * Phi(x) with the exact normal CDF, in fp64."""
    from scipy.special import erf
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def gemm_bf16(a_packed, b_packed, sfa, sfb, M: int, N: int, K: int, alpha: float = 1.0,
              bias: Optional[np.ndarray] = None, residual: Optional[np.ndarray] = None,
              fmt: str = "nvfp4", sf_layout: str = "swizzled", rows=None,
              gelu_act: bool = False) -> GemmResult:
    """alpha * deq(A) @ deq(B)^T (+ bias) (+ residual), rounded to bf16; with
    ``gelu_act``, GELU(alpha * deq(A) @ deq(B)^T + bias) (no residual).

    ``rows`` (optional index array) restricts the result to those rows of the
    output (``residual`` then holds just those rows)."""
    if gelu_act and residual is not None:
        raise ValueError("the GELU epilogue takes no residual")
    a = dequant(a_packed, sfa, M, K, fmt, sf_layout).astype(np.float64)
    b = dequant(b_packed, sfb, N, K, fmt, sf_layout).astype(np.float64)
    if rows is not None:
        a = a[np.asarray(rows)]
        M = a.shape[0]
    alpha64 = float(np.float32(alpha))
    s = a @ b.T
    exact = alpha64 * s
    if bias is not None:
        exact = exact + np.asarray(bias, np.float64).reshape(1, N)
    if residual is not None:
        exact = exact + np.asarray(residual, np.float64).reshape(M, N)
    if gelu_act:
        exact = gelu(exact)
    bound = abs(alpha64) * (np.abs(a) @ np.abs(b).T)
    out = bf16_round(exact.astype(np.float32))
    return GemmResult(exact, out, bound)


def gemm_gelu_nvfp4(a_packed, b_packed, sfa, sfb, M: int, N: int, K: int, alpha: float = 1.0,
                    bias: Optional[np.ndarray] = None, fmt: str = "nvfp4",
                    rows=None) -> OracleResult:
    """GELU(alpha * deq(A) @ deq(B)^T + bias) rounded to fp32 and quantized to
    NVFP4 with tiled scales (rows = output rows, H = N)."""
    g = gemm_bf16(a_packed, b_packed, sfa, sfb, M, N, K, alpha=alpha, bias=bias, fmt=fmt,
                  rows=rows, gelu_act=True)
    return quantize(g.exact.astype(np.float32), "nvfp4", "swizzled")
