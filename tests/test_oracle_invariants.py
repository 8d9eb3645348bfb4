"""Pins for the oracle from invariants and brute force: the scale layout
against the nested tile shape printed on the pages, dequantisation error
bounds, scale-choice optimality and code optimality on tiny rows."""
import numpy as np
import pytest
import torch

import oracle
import workloads

E2M1_VALS = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6],
                     dtype=np.float64)


def _random_case(M, H, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = oracle.round_to_dtype(rng.standard_normal((M, H)).astype(np.float32) * scale, dtype)
    r = oracle.round_to_dtype(rng.standard_normal((M, H)).astype(np.float32) * scale, dtype)
    w = oracle.round_to_dtype((1 + 0.1 * rng.standard_normal(H)).astype(np.float32), dtype)
    return x, r, w


# ---------------------------------------------------------------- layout pins
@pytest.mark.parametrize("M,nb", [(1, 4), (41, 12), (128, 16), (130, 6), (300, 5), (256, 448)])
def test_swizzle_matches_nested_tile_shape(M, nb):
    """The FlashInfer docstring describes the tiled scale buffer as the nested
    shape [m_tile][k_tile][outer_m 32][inner_m 4][inner_k 4] (row-major nesting)
    with outer_m = m % 32 and inner_m = (m % 128) // 32; the vLLM fused_wo_a
    page places tile row r at byte (r % 32) * 16 + (r // 32) * 4.  Build that
    nesting with numpy strides and compare against the oracle's offsets."""
    nkt = (nb + 3) // 4
    mt = (M + 127) // 128
    nested = np.arange(mt * nkt * 512).reshape(mt, nkt, 32, 4, 4)
    m, k = np.meshgrid(np.arange(mt * 128), np.arange(nkt * 4), indexing="ij")
    want = nested[m // 128, k // 4, m % 32, (m % 128) // 32, k % 4]
    got = oracle.swizzled_sf_offset(m, k, nkt)
    assert np.array_equal(got, want)
    # vLLM statement of the in-tile row position, for k % 4 == 0
    r = m % 128
    assert np.array_equal((got % 512)[:, ::4], ((r % 32) * 16 + (r // 32) * 4)[:, ::4])
    # a bijection of the padded grid onto the buffer
    assert np.array_equal(np.sort(got.reshape(-1)), np.arange(mt * nkt * 512))
    assert oracle.sf_size_bytes(M, nb * 16, "nvfp4", "swizzled") == mt * nkt * 512


@pytest.mark.parametrize("M,H,fmt", [(3, 80, "nvfp4"), (129, 160, "mxfp4"), (5, 64, "mxfp4")])
def test_tiled_and_rowmajor_hold_the_same_bytes(M, H, fmt):
    x, r, w = _random_case(M, H, "bf16", 7)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, "bf16", fmt, "both")
    nb = H // oracle.block_size(fmt)
    nkt = (nb + 3) // 4
    m, k = np.meshgrid(np.arange(M), np.arange(nb), indexing="ij")
    assert np.array_equal(o.sf_swizzled[oracle.swizzled_sf_offset(m, k, nkt)],
                          o.sf_rowmajor.reshape(M, nb))
    # every other byte of the tiled buffer is padding and zero
    mask = np.ones(o.sf_swizzled.size, bool)
    mask[oracle.swizzled_sf_offset(m, k, nkt).reshape(-1)] = False
    assert np.all(o.sf_swizzled[mask] == 0)
    assert o.sf_swizzled.size == ((M + 127) // 128) * nkt * 512


# ---------------------------------------------------------------- scale pins
def test_nvfp4_scale_is_nearest_e4m3_to_amax_over_6():
    x, r, w = _random_case(64, 256, "bf16", 11)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, "bf16", "nvfp4", "rowmajor")
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    amax = np.abs(o.y.reshape(64, -1, 16)).max(axis=2).astype(np.float64)
    target = np.minimum(amax / 6.0, 448.0)
    for tgt, code in zip(target.reshape(-1), o.scale_codes.reshape(-1)):
        d = np.abs(vals - tgt)
        best = np.flatnonzero(d <= d.min() * (1 + 1e-6) + 1e-30)
        assert code in best


def test_mxfp4_scale_brackets_amax():
    """MXFP4: the scale is the power of two s with s/2 < amax/6 <= s, so the
    largest element lands in (3, 6] after scaling."""
    x, r, w = _random_case(64, 512, "bf16", 12, scale=3.0)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, "bf16", "mxfp4", "rowmajor")
    amax = np.abs(o.y.reshape(64, -1, 32)).max(axis=2).astype(np.float64)
    ratio = amax / o.scale.astype(np.float64)
    assert np.all(ratio > 3.0) and np.all(ratio <= 6.0 * (1 + 1e-7))
    assert np.all(np.log2(o.scale) == np.round(np.log2(o.scale)))


# ---------------------------------------------------------------- error bounds
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_dequant_error_within_half_step(fmt, dtype):
    """|dequant - y| <= half the E2M1 grid step at |v|, times the scale, when
    |v| <= 6; above 6 (NVFP4 scale rounded down) the error is (|v| - 6) * s."""
    M, H = 32, 1024
    x, r, w = _random_case(M, H, dtype, 13)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, dtype, fmt, "rowmajor")
    deq = oracle.dequant(o.packed, o.sf_rowmajor, M, H, fmt, "rowmajor").astype(np.float64)
    b = oracle.block_size(fmt)
    s = np.repeat(o.scale.astype(np.float64), b, axis=1)
    a = np.abs(o.v.astype(np.float64))
    half_step = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))
    # slack: v is y/s rounded to fp32, so y and v*s differ by <= 1/2 ulp of y
    yabs = np.abs(o.y.astype(np.float64))
    bound = np.where(a <= 6, half_step * s, (a - 6) * s) + yabs * 2.0 ** -23
    err = np.abs(deq - o.y.astype(np.float64))
    assert np.all(err <= bound)
    # and the dequantised values are exactly code value times scale
    assert np.all(np.abs(deq) <= 6 * s)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_codes_are_nearest_by_brute_force_on_tiny_rows(fmt):
    """H = 64: for each element the oracle's code minimises |E2M1(c) * s - y|
    over all 16 codes (exact fp64 search), ties to the even mantissa, the zero
    sign following y.  A mismatch is only allowed where y/s sits within two
    fp32 ulps of an E2M1 midpoint (the oracle scales y by the rounded
    reciprocal of s, then rounds the product to fp32)."""
    x, r, w = _random_case(8, 64, "bf16", 14, scale=2.0)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, "bf16", fmt, "rowmajor")
    b = oracle.block_size(fmt)
    s = np.repeat(o.scale.astype(np.float64), b, axis=1)
    y = o.y.astype(np.float64)
    for i in range(8):
        for j in range(64):
            d = np.abs(E2M1_VALS * s[i, j] - y[i, j])
            best = np.flatnonzero(d == d.min())
            if len(best) > 1:
                mags = {c & 7 for c in best}
                if len(mags) > 1:
                    best = [c for c in best if (c & 1) == 0]
                if len(best) > 1:
                    best = [c for c in best if (c >= 8) == bool(np.signbit(y[i, j]))]
            if o.codes[i, j] != best[0]:
                q = abs(y[i, j] / s[i, j])
                mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
                assert np.min(np.abs(mids - q) / mids) < 2.0 ** -22


# ---------------------------------------------------------------- workloads
def test_workload_generator_is_deterministic_and_sliceable():
    wl = workloads.C3.with_shape(5000, 256)
    a = workloads.make_rows(wl, "x", 0, 5000)
    b = workloads.make_rows(wl, "x", 4090, 4100)
    assert torch.equal(a[4090:4100], b)
    cols = workloads.outlier_columns(wl)
    assert cols.numel() == round(0.01 * 256)
    big = a.float().abs().mean(0)
    assert big[cols].mean() > 20 * big[np.setdiff1d(np.arange(256), cols.numpy())].mean()


def test_algorithmic_bytes_formula():
    # x read + r read + r write (2 B each), H/2 code bytes, H/b scale bytes per
    # layout, weight once.
    assert workloads.C3.algorithmic_bytes() == 383_531_008
    assert workloads.C4.algorithmic_bytes() == 555_755_520
    assert workloads.C1.algorithmic_bytes() == 7_232


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_y_is_one_rounding_of_h_w_rstd(dtype):
    """h * w * rstd is exact in fp64 (8+8+24 or 11+11+24 significant bits), so
    the single-rounding reading of y = (h * w) * rstd means y equals that
    exact product rounded once to fp32, element by element."""
    x, r, w = _random_case(16, 512, dtype, 21, scale=2.0)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, 1e-6, dtype, "nvfp4", "rowmajor")
    exact = (o.residual.astype(np.float64) * w.astype(np.float64)[None, :]) \
        * o.rstd.astype(np.float64)[:, None]
    assert np.array_equal(o.y, exact.astype(np.float32))
