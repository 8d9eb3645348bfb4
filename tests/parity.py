"""Helpers for the GPU-vs-oracle parity tests.

Acceptance rule (stated for this path; the numpy part is tests/acceptance.py):
  * the updated residual is bit-exact;
  * scale bytes and E2M1 codes are bit-exact, except where the oracle's
    pre-rounding value lies within 1e-5 relative of a rounding boundary - an
    E4M3 midpoint or a power of two (UE8M0) for a scale (a flipped scale
    excuses its whole block), an E2M1 midpoint for a code; such exceptions may
    touch at most 1e-4 of the elements;
  * the library's dequantisation of the GPU bytes equals the oracle's
    dequantisation of the same bytes to within 1e-6 of the block scale;
  * every padding byte of the tiled scale buffer is zero.
The GPU side is only ever reached through the C ABI (rmsnorm_fp4_quant_gb300).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq

from acceptance import (  # noqa: F401  (re-exported for the tests)
    BOUNDARY_REL,
    E2M1_MIDS,
    MAX_EXCEPTION_FRAC,
    check_rows,
    e4m3_midpoints,
    near,
    near_pow2,
    tiled_padding_is_zero,
)


@dataclasses.dataclass
class GpuOut:
    rows: np.ndarray          # row ids held below
    residual_bits: np.ndarray # (len(rows), H) uint16
    packed: np.ndarray        # (len(rows), H/2) uint8
    sf: np.ndarray            # whole scale buffer as returned (row-major or tiled), flat
    sf_rm: np.ndarray | None  # whole row-major buffer for layout "both", flat


def run_gpu(x, r, w, eps, fmt, layout, rows=None, stream=None, global_scale=None):
    """x, r, w: CUDA tensors (r is updated in place).  Returns numpy copies
    of the outputs for `rows` (default: every row) and the whole scale
    buffers.  global_scale: optional python float, passed as a device scalar."""
    gs = None if global_scale is None else torch.tensor([global_scale], dtype=torch.float32,
                                                         device=x.device)
    outs = fq.add_rmsnorm_fp4quant(x, r, w, eps=eps, fmt=fmt, sf_layout=layout, stream=stream,
                                   global_scale=gs)
    torch.cuda.synchronize()
    return fetch(outs, r, layout, rows)


def run_quantize(x, fmt, layout, global_scale=None, rows=None):
    gs = None if global_scale is None else torch.tensor([global_scale], dtype=torch.float32,
                                                         device=x.device)
    outs = fq.quantize_fp4(x, fmt=fmt, sf_layout=layout, global_scale=gs)
    torch.cuda.synchronize()
    return fetch(outs, None, layout, rows, M=x.shape[0])


def fetch(outs, r, layout, rows=None, M=None):
    packed, sf = outs[0], outs[1]
    sf_rm = outs[2] if layout == "both" else None
    M = r.shape[0] if M is None else M
    rows = np.arange(M) if rows is None else np.asarray(rows)
    idx = torch.from_numpy(rows).to(packed.device)
    rb = None if r is None else r.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    pk = packed.reshape(M, -1).index_select(0, idx).cpu().numpy()
    return GpuOut(rows, rb, pk, sf.cpu().numpy().reshape(-1),
                  None if sf_rm is None else sf_rm.cpu().numpy().reshape(-1))


def gpu_scale_codes(g: GpuOut, M, H, fmt, layout, rows=None):
    """(len(rows), nb) scale bytes read from the GPU buffer of `layout`."""
    nb = H // oracle.block_size(fmt)
    rows = g.rows if rows is None else np.asarray(rows)
    kk = np.arange(nb)
    if layout == "rowmajor":
        return g.sf.reshape(M, nb)[rows]
    offs = oracle.swizzled_sf_offset(rows[:, None], kk[None, :], (nb + 3) // 4)
    return g.sf[offs]


def compare(g: GpuOut, o: oracle.OracleResult, fmt, layout, dtype, M_full, H,
            check_padding=True):
    """Apply the acceptance rule (tests/acceptance.py) to the GPU rows held in
    `g` against the oracle result `o` computed on exactly those rows, with
    the exception fraction taken over these rows.  Returns a stats dict."""
    rows = g.rows
    assert o.packed.shape[0] == len(rows)
    nb = H // oracle.block_size(fmt)
    g_sc = gpu_scale_codes(g, M_full, H, fmt, "rowmajor" if layout == "rowmajor" else "swizzled",
                           rows)
    n_exc = check_rows(o, g.residual_bits, g_sc, g.packed, fmt, dtype)
    if layout == "both":
        rm = g.sf_rm.reshape(M_full, nb)[rows]
        assert np.array_equal(rm, g_sc), "row-major and tiled scale buffers disagree"
    assert n_exc <= MAX_EXCEPTION_FRAC * o.codes.size, f"{n_exc} exceptions in {o.codes.size}"
    if check_padding and layout in ("swizzled", "both"):
        assert tiled_padding_is_zero(g.sf, M_full, nb), "tiled padding bytes are not zero"
    return {"exceptions": n_exc, "elements": int(o.codes.size)}


def _bits_to_f64(bits, dtype):
    bits = np.asarray(bits, np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def rn16_bits(y_f32, dtype):
    """Bit patterns of fp32 values rounded to nearest-even in bf16 / fp16 (the
    library casts of torch and numpy)."""
    y_f32 = np.ascontiguousarray(y_f32, np.float32)
    if dtype == "bf16":
        return torch.from_numpy(y_f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return y_f32.astype(np.float16).view(np.uint16)


def compare_y(y_bits, y_f32, dtype, rel=BOUNDARY_REL):
    """The y side output against the oracle's fp32 y rounded once to `dtype`.

    y scales with rstd, and the kernel sums h^2 in fp32 in its own order while
    the oracle sums in fp64, so rstd (hence y) may differ by an fp32 ulp or
    two.  That flips the 16-bit rounding only where y sits at a midpoint
    between two 16-bit neighbours.  Accepted: equal bits, or the adjacent
    16-bit value on the other side of a midpoint that y lies within `rel` of.
    Returns the number of excused elements."""
    y_f32 = np.asarray(y_f32, np.float32)
    want = rn16_bits(y_f32, dtype)
    got = np.asarray(y_bits, np.uint16)
    bad = got != want
    if not bad.any():
        return 0
    g, w = got[bad], want[bad]
    same_sign = (g >> 15) == (w >> 15)
    adjacent = same_sign & (np.abs((g & 0x7FFF).astype(np.int32) - (w & 0x7FFF).astype(np.int32)) == 1)
    yv = y_f32[bad].astype(np.float64)
    mid = 0.5 * (_bits_to_f64(g, dtype) + _bits_to_f64(w, dtype))
    at_mid = np.abs(yv - mid) <= rel * np.abs(yv)
    ok = adjacent & at_mid
    idx = np.argwhere(bad)[~ok]
    assert ok.all(), (f"y differs away from a rounding midpoint at {idx[:5].tolist()}: "
                      f"gpu {g[~ok][:5]} oracle {w[~ok][:5]} y {yv[~ok][:5]}")
    assert bad.sum() <= max(1, 1e-3 * bad.size), f"{bad.sum()} excused y elements"
    return int(bad.sum())


def check_dequant(g: GpuOut, M, H, fmt, layout, device="cuda"):
    """The library's dequant of the GPU bytes vs the oracle's dequant of the
    same bytes (every row of the batch must be in `g`)."""
    assert len(g.rows) == M
    lay = "rowmajor" if layout == "rowmajor" else "swizzled"
    packed_t = torch.from_numpy(g.packed).to(device)
    sf_t = torch.from_numpy(g.sf).to(device)
    deq = fq.dequant(packed_t, sf_t, M, H, fmt=fmt, sf_layout=lay)
    torch.cuda.synchronize()
    got = deq.cpu().numpy()
    want = oracle.dequant(g.packed, g.sf, M, H, fmt, lay)
    b = oracle.block_size(fmt)
    nb = H // b
    sc = gpu_scale_codes(g, M, H, fmt, lay)
    s = oracle.e4m3_decode(sc) if oracle.e4m3_scaled(fmt) else oracle.ue8m0_decode(sc)
    tol = np.repeat(s.astype(np.float64), b, axis=1) * 1e-6
    assert np.all(np.abs(got.astype(np.float64) - want) <= tol)
    return got
