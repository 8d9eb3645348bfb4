"""Pins the oracle to hand-derived worked rows (tests/golden/worked_rows.json)
and to closed forms of RMSNorm (a constant row has RMS |c|)."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_rows.json")
ROWS = json.load(open(GOLDEN))["rows"]


def _row_inputs(spec):
    H = spec["H"]
    x = np.full((1, H), spec["x"], np.float32)
    r = np.full((1, H), spec["r"], np.float32)
    if spec["one_hot"]:
        r[:] = 0
        r[0, 0] = 1.0
    w = np.full(H, spec["w"], np.float32)
    return x, r, w


def _check_bytes(arr, spec_bytes):
    for key, val in spec_bytes.items():
        want = int(val, 16)
        if key == "all":
            assert np.all(arr == want), (arr[:8], want)
        elif key == "rest":
            assert np.all(arr[1:] == want), (arr[:8], want)
        else:
            assert arr[int(key)] == want, (key, arr[:8], want)


@pytest.mark.parametrize("spec", ROWS, ids=[r["name"] for r in ROWS])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_worked_row(spec, fmt):
    x, r, w = _row_inputs(spec)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, spec["eps"], spec["dtype"], fmt, "both")
    exp = spec[fmt]
    _check_bytes(o.scale_codes[0], exp["scale_codes"])
    _check_bytes(o.packed[0], exp["bytes"])
    assert abs(float(o.rstd[0]) - spec["rstd"]) <= 2e-7 * spec["rstd"] + 1e-7
    if "residual_bits" in spec:
        bits = (o.residual.view(np.uint32) >> 16).astype(np.uint16)
        assert np.all(bits == int(spec["residual_bits"], 16))
    # both layouts carry the same bytes
    assert np.array_equal(o.sf_rowmajor, o.scale_codes.reshape(-1))


@pytest.mark.parametrize("c", [1.0, -3.0, 0.125, 1000.0, 2.0 ** -6])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_constant_row_rms_closed_form(c, dtype):
    """A constant row c has mean of squares c^2, so rstd = 1/sqrt(c^2 + eps)
    (closed form, fp64) and y = c * rstd * w."""
    H, eps = 128, 1e-6
    x = np.zeros((1, H), np.float32)
    r = np.full((1, H), c, np.float32)
    w = np.linspace(0.5, 1.5, H).astype(np.float32)
    w = oracle.round_to_dtype(w, dtype)
    o = oracle.add_rmsnorm_fp4_quant(x, r, w, eps, dtype, "nvfp4", "rowmajor")
    exact = 1.0 / math.sqrt(c * c + float(np.float32(eps)))
    assert abs(float(o.rstd[0]) - exact) <= 3e-7 * exact
    assert np.allclose(o.y[0], c * exact * w, rtol=4e-7, atol=0)
    # h * w is exact in fp32, so y is within half an ulp of h * w * rstd
    yy = (np.float64(c) * w.astype(np.float64)) * np.float64(o.rstd[0])
    assert np.all(np.abs(o.y[0] - yy) <= np.abs(yy) * 2.0 ** -24)


def test_zero_row_gives_zero_codes_and_scales():
    H = 256
    z = np.zeros((3, H), np.float32)
    w = np.ones(H, np.float32)
    for fmt in ("nvfp4", "mxfp4"):
        o = oracle.add_rmsnorm_fp4_quant(z, z, w, 1e-6, "bf16", fmt, "swizzled")
        assert np.all(o.packed == 0)
        assert np.all(o.scale_codes == 0)
        assert np.all(o.residual == 0)
        assert np.all(o.sf_swizzled == 0)


def test_residual_is_rounded_sum():
    """The new residual is the storage-dtype rounding of x + r (bf16 keeps
    8 significant bits): 1 + 2^-7 is representable, 1 + 2^-8 ties down to 1,
    1 + 3*2^-8 ties up to 1 + 2^-6, 1 + 2^-9 rounds down."""
    H = 64
    x = np.ones((1, H), np.float32)
    r = np.zeros((1, H), np.float32)
    r[0, :4] = [2.0 ** -7, 2.0 ** -8, 3 * 2.0 ** -8, 2.0 ** -9]
    o = oracle.add_rmsnorm_fp4_quant(x, r, np.ones(H, np.float32), 1e-6, "bf16", "nvfp4",
                                     "rowmajor")
    assert o.residual[0, 0] == 1 + 2.0 ** -7
    assert o.residual[0, 1] == 1.0
    assert o.residual[0, 2] == 1 + 2.0 ** -6
    assert o.residual[0, 3] == 1.0


def test_y_side_output_is_y_rounded_once():
    """The optional y output is y rounded to the storage dtype: for the
    constant row, y = 0.99999952 lies between the bf16 neighbours 0.99609375
    and 1.0 and rounds to 1.0; for fp16 (spacing 2^-11 below 1) also to 1.0."""
    for dtype in ("bf16", "fp16"):
        x = np.zeros((1, 64), np.float32)
        r = np.ones((1, 64), np.float32)
        o = oracle.add_rmsnorm_fp4_quant(x, r, np.ones(64, np.float32), 1e-6, dtype, "nvfp4",
                                         "rowmajor")
        assert np.all(o.y_out == 1.0)
        assert np.all(o.y < 1.0)
