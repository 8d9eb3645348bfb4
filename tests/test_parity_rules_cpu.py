"""The acceptance rules of the parity tests, checked on hand-made cases so that
a GPU run can trust them: a y element may differ from the oracle's only by one
16-bit ulp, and only where the oracle's fp32 y sits at a rounding midpoint."""
import numpy as np
import pytest

import parity


def _y(vals):
    return np.array(vals, np.float32).reshape(1, -1)


def _bits(vals, dtype):
    """Exact 16-bit patterns of values that are representable in `dtype`."""
    a = np.array(vals, np.float64)
    if dtype == "bf16":
        b = (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), a)
    else:
        b = a.astype(np.float16).view(np.uint16)
        assert np.array_equal(b.view(np.float16).astype(np.float64), a)
    return b.reshape(1, -1)


# (midpoint between two 16-bit neighbours, the lower neighbour, the upper one)
MIDS = {"bf16": (1.0 + 2.0 ** -8, 1.0, 1.0 + 2.0 ** -7),
        "fp16": (1.0 + 2.0 ** -11, 1.0, 1.0 + 2.0 ** -10)}


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_y_rounded_to_nearest_pass(dtype):
    """Values a quarter and three quarters of an ulp above a 16-bit number,
    of both signs: the expected bits are the nearest neighbour, not the
    truncation."""
    mid, lo, hi = MIDS[dtype]
    q = 0.25 * (hi - lo)
    vals = [lo + q, lo + 3 * q, -(lo + q), -(lo + 3 * q)]
    want = [lo, hi, -lo, -hi]
    assert parity.compare_y(_bits(want, dtype), _y(vals), dtype) == 0
    with pytest.raises(AssertionError):
        parity.compare_y(_bits([lo, lo, -lo, -lo], dtype), _y(vals), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_y_flip_at_midpoint_excused(dtype, sign):
    mid, lo, hi = MIDS[dtype]
    y = _y([sign * mid] + [0.5] * 3000)
    got = _bits([sign * hi] + [0.5] * 3000, dtype)      # the oracle rounds to even: lo
    assert parity.compare_y(got, y, dtype) == 1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_y_flip_away_from_midpoint_rejected(dtype):
    mid, lo, hi = MIDS[dtype]
    y = _y([lo + 0.25 * (hi - lo)] + [0.5] * 3000)     # a quarter ulp: rounds to lo
    with pytest.raises(AssertionError, match="away from a rounding midpoint"):
        parity.compare_y(_bits([hi] + [0.5] * 3000, dtype), y, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_y_two_ulp_or_sign_flip_rejected(dtype):
    mid, lo, hi = MIDS[dtype]
    y = _y([mid] + [0.5] * 3000)
    two_up = hi + (hi - lo)
    with pytest.raises(AssertionError):
        parity.compare_y(_bits([two_up] + [0.5] * 3000, dtype), y, dtype)
    with pytest.raises(AssertionError):
        parity.compare_y(_bits([-lo] + [0.5] * 3000, dtype), y, dtype)


def test_y_too_many_excused_rejected():
    mid, lo, hi = MIDS["bf16"]
    y = _y([mid] * 10 + [0.5] * 10)
    with pytest.raises(AssertionError, match="excused y elements"):
        parity.compare_y(_bits([hi] * 10 + [0.5] * 10, "bf16"), y, "bf16")
