"""Helpers for the GPU-vs-oracle parity tests.

Acceptance rule (stated for this path):
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

BOUNDARY_REL = 1e-5
MAX_EXCEPTION_FRAC = 1e-4
E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_E4M3_VALS = None


def e4m3_midpoints():
    global _E4M3_VALS
    if _E4M3_VALS is None:
        vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
        _E4M3_VALS = (vals[:-1] + vals[1:]) / 2
    return _E4M3_VALS


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
    """Apply the acceptance rule to the GPU rows held in `g` against the
    oracle result `o` computed on exactly those rows.  Returns a stats dict."""
    rows = g.rows
    assert o.packed.shape[0] == len(rows)
    b = oracle.block_size(fmt)
    nb = H // b
    # 1. residual (the standalone quantize has none)
    if g.residual_bits is not None:
        want_bits = (o.residual.view(np.uint32) >> 16).astype(np.uint16) if dtype == "bf16" \
            else o.residual.astype(np.float16).view(np.uint16)
        bad_res = np.argwhere(g.residual_bits != want_bits)
        assert bad_res.size == 0, f"residual differs at {bad_res[:5].tolist()}"

    # 2. scales
    g_sc = gpu_scale_codes(g, M_full, H, fmt, "rowmajor" if layout == "rowmajor" else "swizzled",
                           rows)
    sc_bad = g_sc != o.scale_codes
    if oracle.e4m3_scaled(fmt):
        sc_excusable = near(o.t, e4m3_midpoints())
    else:
        sc_excusable = near_pow2(o.t)
    unexcused = sc_bad & ~sc_excusable
    assert not unexcused.any(), (
        f"scale bytes differ away from a boundary at {np.argwhere(unexcused)[:5].tolist()}: "
        f"gpu {g_sc[unexcused][:5]} oracle {o.scale_codes[unexcused][:5]} t {o.t[unexcused][:5]}")
    if layout == "both":
        rm = g.sf_rm.reshape(M_full, nb)[rows]
        assert np.array_equal(rm, g_sc), "row-major and tiled scale buffers disagree"

    # 3. codes
    g_codes = np.empty((len(rows), H), np.uint8)
    pk = g.packed
    g_codes[:, 0::2] = pk & 0xF
    g_codes[:, 1::2] = pk >> 4
    code_bad = g_codes != o.codes
    block_excused = np.repeat(sc_bad, b, axis=1)
    code_excusable = near(np.abs(o.v), E2M1_MIDS) | block_excused
    unexcused = code_bad & ~code_excusable
    assert not unexcused.any(), (
        f"codes differ away from a boundary at {np.argwhere(unexcused)[:5].tolist()}: "
        f"gpu {g_codes[unexcused][:8]} oracle {o.codes[unexcused][:8]} v {o.v[unexcused][:8]}")
    n_exc = int(code_bad.sum() + sc_bad.sum())
    assert n_exc <= MAX_EXCEPTION_FRAC * o.codes.size, f"{n_exc} exceptions in {o.codes.size}"

    # 4. tiled padding
    if check_padding and layout in ("swizzled", "both"):
        nkt = (nb + 3) // 4
        mask = np.ones(g.sf.size, bool)
        mm, kk = np.meshgrid(np.arange(M_full), np.arange(nb), indexing="ij")
        mask[oracle.swizzled_sf_offset(mm, kk, nkt).reshape(-1)] = False
        assert np.all(g.sf[mask] == 0), "tiled padding bytes are not zero"
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
