"""Number formats used by the oracle: bf16/fp16 rounding, E2M1, E4M3, UE8M0.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The FlashInfer page (``add_rmsnorm_fp4quant.py``) imports its conversions
(``cvt_f32_to_e4m3``, ``cvt_f32_to_ue8m0``, ``quantize_and_pack_16`` ...) from a
helper module whose bodies are not on the page; its Notes give only the
format maxima (E2M1 max 6.0, E4M3 max 448.0, UE8M0 = powers of two).  The
rounding rules below are therefore the stated readings:

  * E2M1 codes: round to nearest on the grid {0, .5, 1, 1.5, 2, 3, 4, 6}, ties
    to the even grid index (= even mantissa bit), magnitudes above 6 saturate
    to 6, sign kept as the top bit of the nibble (sign-magnitude);
  * E4M3 scales: round to nearest, ties to even mantissa, subnormals down to
    2^-9, never NaN (inputs are clamped to <= 448 first);
  * UE8M0 scales: the power of two at or above the value (ceil of log2),
    exponent clamped to [-127, 127], code = exponent + 127 (0xFF never made).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# E2M1 magnitudes by 3-bit index: exponent bits ee, mantissa bit m -> (ee m).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


# ----------------------------------------------------------------------------
# storage dtypes
# ----------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even), returned as fp32.

    bf16 keeps the top 16 bits of the fp32 encoding; the discarded low half is
    rounded with the usual bias trick (add 0x7FFF plus the kept LSB).  Finite
    inputs only (the workloads have no NaN).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return (rounded.astype(np.uint32) << np.uint32(16)).view(np.float32)


def fp16_round(a) -> np.ndarray:
    """Round fp32 values to IEEE half (nearest, ties to even), returned as fp32."""
    return np.asarray(a, dtype=np.float32).astype(np.float16).astype(np.float32)


def round_to_dtype(a, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_round(a)
    if dtype == "fp16":
        return fp16_round(a)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# E2M1 (FP4) element codes
# ----------------------------------------------------------------------------
def e2m1_index_rne(a) -> np.ndarray:
    """3-bit grid index nearest to magnitude ``a`` (>= 0), ties to even index.

    Values above 6 land on index 7 (saturation).  Walks the seven midpoints
    between neighbouring grid values: above a midpoint -> the upper index;
    exactly on it -> whichever of the two indices is even.
    """
    a = np.asarray(a, dtype=np.float32)
    idx = np.zeros(a.shape, dtype=np.uint8)
    for i in range(7):
        mid = (E2M1_GRID[i] + E2M1_GRID[i + 1]) / F32(2)   # exact in fp32
        upper = i + 1
        on_tie_pick = upper if upper % 2 == 0 else i
        idx = np.where(a > mid, np.uint8(upper), idx)
        idx = np.where(a == mid, np.uint8(on_tie_pick), idx)
    return idx.astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """4-bit code of fp32 ``v``: sign bit 3, grid index bits 0-2."""
    v = np.asarray(v, dtype=np.float32)
    idx = e2m1_index_rne(np.abs(v))
    sign = np.signbit(v).astype(np.uint8)
    return (sign << np.uint8(3)) | idx


def e2m1_decode(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.uint8)
    mag = E2M1_GRID[code & np.uint8(7)]
    return np.where((code & np.uint8(8)) != 0, -mag, mag).astype(np.float32)


# ----------------------------------------------------------------------------
# E4M3 (OCP FP8, "fn" variant: no infinities, 0x7F/0xFF are NaN)
# ----------------------------------------------------------------------------
def e4m3_decode(code) -> np.ndarray:
    """fp32 value of each E4M3 byte: bias 7, 3 mantissa bits, subnormals at
    exponent field 0, S.1111.111 is NaN."""
    code = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(code & 0x80, -1.0, 1.0)
    e = (code >> 3) & 0xF
    m = code & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e.astype(np.float64) - 10))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return (sign * mag).astype(np.float32)


def e4m3_encode_rne(t) -> np.ndarray:
    """E4M3 code nearest to ``t`` (0 <= t <= 448), ties to even mantissa.

    The quantum of the binade holding t is 2^(floor(log2 t) - 3), but never
    below the subnormal quantum 2^-9.  t / quantum is an exact fp64 number;
    ``np.rint`` rounds it half-to-even, which is the mantissa's parity.
    """
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    if np.any(t < 0) or np.any(t > 448) or np.any(np.isnan(t)):
        raise ValueError("e4m3_encode_rne expects 0 <= t <= 448")
    safe = np.where(t > 0, t, 1.0)
    _, k = np.frexp(safe)                       # safe = f * 2^k, f in [0.5, 1)
    e = np.maximum(k - 1, -6)                   # binade exponent, subnormal floor
    q = np.exp2((e - 3).astype(np.float64))
    n = np.rint(t / q)                          # exact quotient, half-to-even
    val = n * q                                 # the chosen E4M3 value (exact)
    # encode val
    _, kv = np.frexp(np.where(val > 0, val, 1.0))
    ev = kv - 1
    sub = val < 2.0 ** -6
    mant_sub = np.rint(val / 2.0 ** -9)
    mant_norm = np.rint(val / np.exp2(ev.astype(np.float64)) * 8) - 8
    code = np.where(sub, mant_sub, ((ev + 7) << 3) + mant_norm)
    code = np.where(t > 0, code, 0)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------
# UE8M0 (unsigned exponent-only byte)
# ----------------------------------------------------------------------------
def ue8m0_encode_ceil(t) -> np.ndarray:
    """Code of the smallest power of two >= t (t >= 0), exponent clamped to
    [-127, 127]; t == 0 gives code 0 (2^-127)."""
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    if np.any(t < 0) or np.any(np.isnan(t)):
        raise ValueError("ue8m0_encode_ceil expects t >= 0")
    safe = np.where(t > 0, t, 1.0)
    f, k = np.frexp(safe)                       # safe = f * 2^k, f in [0.5, 1)
    e = np.where(f == 0.5, k - 1, k)            # exact power of two: no step up
    e = np.where(t > 0, e, -127)
    e = np.clip(e, -127, 127)
    return (e + 127).astype(np.uint8)


def ue8m0_decode(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.uint8).astype(np.float64)
    val = np.exp2(code - 127.0)
    val = np.where(code == 255, np.nan, val)
    return val.astype(np.float32)
