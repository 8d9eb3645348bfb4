"""The acceptance rule of the GPU-vs-oracle parity tests on numpy arrays alone
(no torch, no GPU), so that spawned worker processes can apply it to blocks of
rows of a full-size workload.

Rule (stated for this path):
  * the updated residual is bit-exact;
  * scale bytes and E2M1 codes are bit-exact, except where the oracle's
    pre-rounding value lies within 1e-5 relative of a rounding boundary - an
    E4M3 midpoint or a power of two (UE8M0) for a scale (a flipped scale
    excuses its whole block), an E2M1 midpoint for a code; such exceptions may
    touch at most 1e-4 of the elements of a workload (the caller sums them
    over all of its rows before applying the fraction);
  * every padding byte of the tiled scale buffer is zero.
"""
from __future__ import annotations

import numpy as np

import oracle

BOUNDARY_REL = 1e-5
MAX_EXCEPTION_FRAC = 1e-4
E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_E4M3_MIDS = None


def e4m3_midpoints():
    global _E4M3_MIDS
    if _E4M3_MIDS is None:
        vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
        _E4M3_MIDS = (vals[:-1] + vals[1:]) / 2
    return _E4M3_MIDS


def near(values, bounds, rel=BOUNDARY_REL):
    """True where a value lies within `rel` (relative) of any boundary."""
    v = np.abs(np.asarray(values, np.float64)).reshape(-1)
    b = np.asarray(bounds, np.float64)
    i = np.clip(np.searchsorted(b, v), 1, len(b) - 1)
    d = np.minimum(np.abs(v - b[i - 1]), np.abs(v - b[i]))
    return (d <= rel * np.maximum(v, 1e-30)).reshape(np.shape(values))


def near_pow2(values, rel=BOUNDARY_REL):
    v = np.asarray(values, np.float64)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(v > 0, v, 1.0))
    nearest = np.exp2(np.round(lg))
    return (np.abs(v - nearest) <= rel * v) & (v > 0)


def unpack_codes(packed):
    """(rows, H/2) bytes -> (rows, H) codes, element 2j in the low nibble."""
    packed = np.asarray(packed, np.uint8)
    codes = np.empty((packed.shape[0], 2 * packed.shape[1]), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    return codes


def residual_bits(o_residual, dtype):
    """The 16-bit patterns of the oracle's residual (fp32 values exact in dtype)."""
    if dtype == "bf16":
        return (np.asarray(o_residual, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return np.asarray(o_residual, np.float32).astype(np.float16).view(np.uint16)


def check_rows(o, res_bits, scale_bytes, packed, fmt, dtype):
    """The rule on one set of rows: `o` is the oracle's result on them;
    res_bits (uint16, or None for the standalone quantize), scale_bytes
    (rows, nb) as read from the GPU's buffer, packed (rows, H/2) the GPU's
    codes.  Raises on a difference the rule does not excuse; returns the number
    of excused exceptions (scale bytes + codes).  The exception fraction is
    the caller's to apply, over a whole workload."""
    b = oracle.block_size(fmt)
    if res_bits is not None:
        bad_res = np.argwhere(np.asarray(res_bits, np.uint16) != residual_bits(o.residual, dtype))
        assert bad_res.size == 0, f"residual differs at {bad_res[:5].tolist()}"
    g_sc = np.asarray(scale_bytes, np.uint8)
    sc_bad = g_sc != o.scale_codes
    sc_excusable = near(o.t, e4m3_midpoints()) if oracle.e4m3_scaled(fmt) else near_pow2(o.t)
    unexcused = sc_bad & ~sc_excusable
    assert not unexcused.any(), (
        f"scale bytes differ away from a boundary at {np.argwhere(unexcused)[:5].tolist()}: "
        f"gpu {g_sc[unexcused][:5]} oracle {o.scale_codes[unexcused][:5]} t {o.t[unexcused][:5]}")
    g_codes = unpack_codes(packed)
    code_bad = g_codes != o.codes
    code_excusable = near(np.abs(o.v), E2M1_MIDS) | np.repeat(sc_bad, b, axis=1)
    unexcused = code_bad & ~code_excusable
    assert not unexcused.any(), (
        f"codes differ away from a boundary at {np.argwhere(unexcused)[:5].tolist()}: "
        f"gpu {g_codes[unexcused][:8]} oracle {o.codes[unexcused][:8]} v {o.v[unexcused][:8]}")
    return int(code_bad.sum() + sc_bad.sum())


def bits_to_f32(bits, dtype):
    """16-bit storage patterns -> their exact fp32 values."""
    bits = np.asarray(bits, np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def fused_block_task(args):
    """Worker task: the oracle on one block of rows of the fused op and the
    rule against the GPU's bytes for them; returns (exceptions, elements)."""
    x_bits, r_bits, w, eps, dtype, fmt, res_bits, packed, scale_bytes = args
    x = bits_to_f32(x_bits, dtype)
    r = bits_to_f32(r_bits, dtype)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, eps, dtype, fmt, "rowmajor")
    n = check_rows(o, res_bits, scale_bytes, packed, fmt, dtype)
    return n, int(o.codes.size)


def tiled_padding_is_zero(sf, M, nb):
    """Every byte of a 128x4 tiled scale buffer outside the M x nb scales is 0.
    The buffer is [m/128][k/4][m%32][(m%128)/32][k%4] in C order."""
    nkt = (nb + 3) // 4
    mt = (M + 127) // 128
    t = np.asarray(sf, np.uint8).reshape(mt, nkt, 32, 4, 4)
    m = (np.arange(mt)[:, None, None, None, None] * 128 +
         np.arange(32)[None, None, :, None, None] + np.arange(4)[None, None, None, :, None] * 32)
    k = np.arange(nkt)[None, :, None, None, None] * 4 + np.arange(4)[None, None, None, None, :]
    pad = np.broadcast_to((m >= M) | (k >= nb), t.shape)
    return bool(np.all(t[pad] == 0))


def quantize_block_task(args):
    """Worker task: the oracle's standalone quantize on one block of rows and
    the rule against the GPU's bytes for them; returns (exceptions, elements)."""
    x_bits, dtype, fmt, packed, scale_bytes = args
    o = oracle.quantize(bits_to_f32(x_bits, dtype), fmt, "rowmajor")
    n = check_rows(o, None, scale_bytes, packed, fmt, dtype)
    return n, int(o.codes.size)


def gemm_block_bits_task(args):
    """Worker task: the GEMM oracle's bf16 output bits for one block of rows
    (its A rows and their tiled scales are passed alone; a block starts on a
    128-row tile, so its scales are a contiguous slice of the tiled buffer)."""
    a, b, sfa, sfb, M, N, K, fmt = args
    g = oracle.gemm_bf16(a, b, sfa, sfb, M, N, K, fmt=fmt)
    return (np.asarray(g.out, np.float32).view(np.uint32) >> 16).astype(np.uint16)
