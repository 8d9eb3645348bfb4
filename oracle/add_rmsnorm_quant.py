"""Oracle of the fused op: residual add, RMSNorm, block-scaled FP4 quantization.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the FlashInfer page ``add_rmsnorm_fp4quant.py``: the module docstring
(residual updated in place to input + residual, y = residual / sqrt(mean of
squares + eps) * weight, then FP4 quantization) and ``kernel`` phases 2 and 3,
written as the plain per-row definition with the rounding rule of
``oracle.formats``.  Per row m (fp32, each op rounded to nearest even):

  1. h = round_dtype(float(x) + float(r))            (phase 2; new residual)
  2. ss = sum of h^2 in fp64;  ms = fp32(ss / H);  rstd = 1 / sqrt(ms + eps)
  3. y = (h * w) * rstd   (h * w of two 16-bit values is exact in fp32, so
     y is the single rounding of h * w * rstd)
  4. per block of b elements: amax = max |y|
       E4M3 scales (NVFP4, b = 16; or b = 32 with E4M3 forced):
           t = min((gs * amax) / 6, 448),  scale = E4M3_rne(t)
       UE8M0 scales (MXFP4, b = 32):
           t = amax / 6,  scale = UE8M0 at or above t   (gs not applied)
  5. inv = (1 / s) * gs for E4M3 scales, 1 / s for UE8M0 (each op rounded to
     nearest fp32);  v = y * inv;  code = E2M1_rne(v)   (s == 0: codes 0)
  6. two codes per byte, element 2j in the low nibble
  (side output, on request: y rounded to nearest-even in the storage dtype)
  7. scale bytes row-major [m, k] and/or in the 128x4 tile order
     (m//128)*nkt*512 + (k//4)*512 + (m%32)*16 + ((m%128)//32)*4 + k%4,
     nkt = ceil(nb / 4), every padding byte of the tiled buffer zero.

Readings where the pages are silent (helper bodies absent):
  * the sum of squares uses the rounded h (the value written back), fp64 sum;
  * y multiplies h by w first and then by rstd, the order of the page's
    cluster branch (``bfloat2_mul_8(h, w)`` then the product times rstd,
    ``max_abs = max_xw * rstd``), without its rounding of h * w to 16 bits:
    the product of two bf16/fp16 values is exact in fp32, so y carries one
    rounding only;
  * the page scales y by the reciprocal of the decoded block scale
    (``fp8_e4m3_to_f32_and_rcp`` / ``ue8m0_to_output_scale`` feeding
    ``quantize_and_pack_16`` in kernel phase 3) without saying how the
    reciprocal is rounded; here it is the correctly rounded fp32 reciprocal,
    then one rounded product (for MXFP4 the reciprocal of a power of two is
    exact, so v is the correctly rounded quotient);
  * a block whose scale is zero (amax = 0, or NVFP4 amax/6 below half the
    smallest E4M3 subnormal) gets all-zero codes;
  * padding rows [M, 128*ceil(M/128)) and padding k in [nb, 4*nkt) of the
    tiled buffer are written 0 (the vLLM ``fused_wo_a`` page zero-fills its
    own padding in the same tile order);
  * global scale gs (the page's ``global_scale``, one fp32 read on the
    device, default 1): the kernel code multiplies it into the E4M3 scale
    (``global_scale_val * max_abs * fp4_max_rcp``) and into the reciprocal
    (``fp8_e4m3_to_f32_and_rcp(...) * global_scale_val``); the docstring's
    "divided by global_scale" is not what the code computes, so the code is
    followed: with gs = 448 * 6 / amax_tensor the block scales use the E4M3
    range and a consumer divides by gs.  UE8M0 scales ignore gs, as on the
    page;
  * ``scale_format="e4m3"`` with 32-element blocks (the page's
    ``scale_format`` on its block-32 branch) is format "e4m3b32": MXFP4
    blocking with NVFP4-style scales.

``quantize`` is the same steps 4-7 applied to an input without the residual
add and the normalisation (y = x), the standalone producer of the FlashRT
``fp4-gemm`` README (``quantize_fp4_sfa_bf16`` / ``_fp16``).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from .formats import (
    F32,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode_rne,
    round_to_dtype,
    ue8m0_decode,
    ue8m0_encode_ceil,
)

E2M1_MAX = F32(6.0)      # FlashInfer page, Notes: FP4 E2M1 maximum
E4M3_MAX = F32(448.0)    # FlashInfer page, Notes: E4M3 maximum


def block_size(fmt: str) -> int:
    return {"nvfp4": 16, "mxfp4": 32, "e4m3b32": 32}[fmt]


def e4m3_scaled(fmt: str) -> bool:
    """True for the formats with E4M3 block scales (global scale applies)."""
    return fmt in ("nvfp4", "e4m3b32")


def swizzled_sf_offset(m, k, nkt):
    """Byte offset of scale (row m, block k) in the 128x4 tiled layout
    (FlashInfer page, ``add_rmsnorm_fp4quant`` Parameters,
    ``is_sf_swizzled_layout``; same in-tile order in vLLM ``fused_wo_a``)."""
    m = np.asarray(m, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    return ((m // 128) * nkt * 512 + (k // 4) * 512 + (m % 32) * 16
            + ((m % 128) // 32) * 4 + (k % 4))


def sf_size_bytes(M: int, H: int, fmt: str, layout: str) -> int:
    """Bytes of one scale buffer (FlashInfer page, output allocation:
    row-major (M, H/b); tiled ceil(M/128) * ceil((H/b)/4) * 512)."""
    nb = H // block_size(fmt)
    if layout == "rowmajor":
        return M * nb
    if layout == "swizzled":
        return ((M + 127) // 128) * ((nb + 3) // 4) * 512
    raise ValueError(layout)


@dataclasses.dataclass
class OracleResult:
    residual: np.ndarray          # (M, H) fp32 holding dtype values: new residual
    packed: np.ndarray            # (M, H/2) uint8
    scale_codes: np.ndarray       # (M, nb) uint8, row-major
    sf_rowmajor: Optional[np.ndarray]   # (M*nb,) uint8 when asked
    sf_swizzled: Optional[np.ndarray]   # tiled buffer when asked
    codes: np.ndarray             # (M, H) uint8 4-bit codes
    rstd: np.ndarray              # (M,) fp32
    y: np.ndarray                 # (M, H) fp32 normalised, weighted
    t: np.ndarray                 # (M, nb) fp32 value the scale rounds from
    scale: np.ndarray             # (M, nb) fp32 decoded scale
    v: np.ndarray                 # (M, H) fp32 value each code rounds from
    y_out: Optional[np.ndarray] = None   # (M, H) y rounded to the storage dtype (fused op)


def add_rmsnorm_fp4_quant(x, r, w, eps: float, dtype: str, fmt: str,
                          layout: str, global_scale: float = 1.0) -> OracleResult:
    """Run the oracle on one batch.

    x, r: (M, H) arrays of dtype values (any float type; converted exactly to
    fp32); w: (H,); dtype "bf16"/"fp16"; fmt "nvfp4"/"mxfp4"/"e4m3b32";
    layout "rowmajor", "swizzled" or "both"; global_scale a positive fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    r = np.asarray(r, dtype=np.float32)
    w = np.asarray(w, dtype=np.float32)
    M, H = x.shape
    b = block_size(fmt)
    if H % b or H < 64:
        raise ValueError("H must be a multiple of the block size and >= 64")

    # 1. residual add, rounded to the storage dtype
    h = round_to_dtype(x + r, dtype)

    # 2. mean of squares and reciprocal root
    ss = np.sum(h.astype(np.float64) ** 2, axis=1)
    ms = (ss / H).astype(np.float32)
    rstd = F32(1.0) / np.sqrt(ms + F32(eps))

    # 3. weight, then normalise (h * w is exact in fp32)
    y = (h * w[None, :]) * rstd[:, None]
    res = _quantize_rows(y, h, rstd, fmt, layout, global_scale)
    # optional side output: y itself rounded once to the storage dtype
    res.y_out = round_to_dtype(y, dtype)
    return res


def quantize(x, fmt: str, layout: str, global_scale: float = 1.0) -> OracleResult:
    """Steps 4-7 on x itself (no add, no normalisation): the standalone
    producer.  `residual` and `rstd` of the result are x and ones."""
    x = np.asarray(x, dtype=np.float32)
    M, H = x.shape
    if H % block_size(fmt) or H < 16:
        raise ValueError("H must be a multiple of the block size")
    return _quantize_rows(x.copy(), x, np.ones(M, np.float32), fmt, layout, global_scale)


def _quantize_rows(y, h, rstd, fmt, layout, global_scale) -> OracleResult:
    M, H = y.shape
    b = block_size(fmt)
    nb = H // b
    gs = F32(global_scale)

    # 4. per-block amax and scale
    yb = y.reshape(M, nb, b)
    amax = np.max(np.abs(yb), axis=2) if M else np.zeros((0, nb), np.float32)
    if e4m3_scaled(fmt):
        t = np.minimum((gs * amax) / E2M1_MAX, E4M3_MAX)
        scode = e4m3_encode_rne(t)
        scale = e4m3_decode(scode)
    else:
        t = amax / E2M1_MAX
        scode = ue8m0_encode_ceil(t)
        scale = ue8m0_decode(scode)

    # 5. element codes: y times the rounded reciprocal of the scale (times gs
    #    for E4M3 scales)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = (F32(1.0) / scale).astype(np.float32)
        if e4m3_scaled(fmt):
            inv = (inv * gs).astype(np.float32)
        vb = yb * inv[:, :, None]
    vb = np.where(scale[:, :, None] == 0, F32(0.0), vb).astype(np.float32)
    v = vb.reshape(M, H)
    codes = e2m1_encode(v)

    # 6. pack, element 2j in the low nibble
    packed = (codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))).astype(np.uint8)

    # 7. scale layouts
    sf_rm = scode.reshape(-1).copy() if layout in ("rowmajor", "both") else None
    sf_sw = None
    if layout in ("swizzled", "both"):
        nkt = (nb + 3) // 4
        sf_sw = np.zeros(sf_size_bytes(M, H, fmt, "swizzled"), dtype=np.uint8)
        mm, kk = np.meshgrid(np.arange(M), np.arange(nb), indexing="ij")
        sf_sw[swizzled_sf_offset(mm, kk, nkt)] = scode
    return OracleResult(h, packed, scode, sf_rm, sf_sw, codes, rstd, y, t, scale, v)


def dequant(packed, sf, M: int, H: int, fmt: str, layout: str) -> np.ndarray:
    """E2M1 value times its block scale, fp32 (exact), from packed bytes and a
    scale buffer in either layout (FlashRT ``fp4-gemm`` README, Validation:
    compare through the dequantised values).  With a global scale gs the
    original values are approximately this divided by gs."""
    packed = np.asarray(packed, dtype=np.uint8).reshape(M, H // 2)
    b = block_size(fmt)
    nb = H // b
    codes = np.empty((M, H), dtype=np.uint8)
    codes[:, 0::2] = packed & np.uint8(0xF)
    codes[:, 1::2] = packed >> np.uint8(4)
    sf = np.asarray(sf, dtype=np.uint8).reshape(-1)
    mm, kk = np.meshgrid(np.arange(M), np.arange(nb), indexing="ij")
    if layout == "rowmajor":
        scode = sf[mm * nb + kk]
    else:
        scode = sf[swizzled_sf_offset(mm, kk, (nb + 3) // 4)]
    scale = e4m3_decode(scode) if e4m3_scaled(fmt) else ue8m0_decode(scode)
    vals = e2m1_decode(codes).reshape(M, nb, b) * scale[:, :, None]
    return vals.reshape(M, H).astype(np.float32)
