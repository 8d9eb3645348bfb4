"""Pins for the global scale, E4M3 scales on 32-element blocks and the
standalone quantize: hand-derived rows (tests/golden/global_scale_and_quantize.json),
brute-force scale choice, and invariants."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "global_scale_and_quantize.json")
ROWS = json.load(open(GOLDEN))["rows"]


def _run(spec):
    H = spec["H"]
    if spec["op"] == "quantize":
        x = np.full((1, H), spec["x"], np.float32)
        return oracle.quantize(x, spec["fmt"], "both", spec["gs"])
    x = np.full((1, H), spec["x"], np.float32)
    r = np.full((1, H), spec["r"], np.float32)
    if spec["op"] == "fused_one_hot":
        r[:] = 0
        r[0, 0] = 1.0
    w = np.ones(H, np.float32)
    return oracle.add_rmsnorm_fp4_quant(x, r, w, spec["eps"], spec["dtype"], spec["fmt"], "both",
                                        spec["gs"])


def _check(arr, spec):
    for key, val in spec.items():
        want = int(val, 16)
        if key == "all":
            assert np.all(arr == want), (arr[:8], want)
        elif key == "rest":
            assert np.all(arr[1:] == want)
        else:
            assert arr[int(key)] == want


@pytest.mark.parametrize("spec", ROWS, ids=[r["name"] for r in ROWS])
def test_golden_row(spec):
    o = _run(spec)
    _check(o.scale_codes[0], spec["scale_codes"])
    _check(o.packed[0], spec["bytes"])
    if "n_scales" in spec:
        assert o.scale_codes.shape[1] == spec["n_scales"]


def _rand(M, H, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, H)) * scale).astype(np.float32)


@pytest.mark.parametrize("fmt,gs", [("nvfp4", 2688.0 / 7.3), ("e4m3b32", 3.7), ("e4m3b32", 1.0)])
def test_e4m3_scale_is_nearest_to_gs_amax_over_6(fmt, gs):
    x = _rand(32, 256, 1, 3.0)
    o = oracle.quantize(x, fmt, "rowmajor", gs)
    b = oracle.block_size(fmt)
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    amax = np.abs(x.reshape(32, -1, b)).max(axis=2).astype(np.float64)
    target = np.minimum(np.float32(gs) * amax / 6.0, 448.0)
    for tgt, code in zip(target.reshape(-1), o.scale_codes.reshape(-1)):
        d = np.abs(vals - tgt)
        assert code in np.flatnonzero(d <= d.min() * (1 + 1e-6) + 1e-30)


@pytest.mark.parametrize("fmt", ["nvfp4", "e4m3b32"])
def test_global_scale_dequant_recovers_values(fmt):
    """With gs = 448*6/amax(tensor) every block scale lies in the E4M3 range and
    dequant / gs is within half a grid step (times s / gs) of x."""
    x = _rand(16, 512, 2, 5.0)
    gs = np.float32(448.0 * 6.0 / np.abs(x).max())
    o = oracle.quantize(x, fmt, "rowmajor", float(gs))
    deq = oracle.dequant(o.packed, o.sf_rowmajor, 16, 512, fmt, "rowmajor").astype(np.float64)
    b = oracle.block_size(fmt)
    s = np.repeat(o.scale.astype(np.float64), b, axis=1) / float(gs)
    a = np.abs(o.v.astype(np.float64))
    half = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))
    bound = np.where(a <= 6, half * s, (a - 6) * s) + np.abs(x) * 2.0 ** -21
    assert np.all(np.abs(deq / float(gs) - x) <= bound)
    assert o.scale_codes.max() <= 0x7E


def test_ue8m0_ignores_global_scale():
    x = _rand(8, 256, 3)
    a = oracle.quantize(x, "mxfp4", "both", 1.0)
    b = oracle.quantize(x, "mxfp4", "both", 37.0)
    assert np.array_equal(a.packed, b.packed) and np.array_equal(a.sf_swizzled, b.sf_swizzled)


def test_quantize_is_the_fused_op_on_unit_rms_rows():
    """A row with mean square exactly 1 (entries +-1), residual 0, weight 1 and
    eps 0 has rstd = 1 exactly, so the fused op quantizes x itself."""
    rng = np.random.default_rng(4)
    x = np.where(rng.random((6, 128)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[:, ::7] *= 0.5          # keep values exact in bf16; fix the RMS below
    x[:, ::7] = np.sign(x[:, ::7])
    q = oracle.quantize(x, "nvfp4", "both")
    f = oracle.add_rmsnorm_fp4_quant(x, np.zeros_like(x), np.ones(128, np.float32), 0.0,
                                     "bf16", "nvfp4", "both")
    assert np.all(f.rstd == 1.0)
    assert np.array_equal(q.packed, f.packed) and np.array_equal(q.sf_swizzled, f.sf_swizzled)
