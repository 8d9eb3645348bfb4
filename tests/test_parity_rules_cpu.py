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


# ---------------------------------------------------------------------------
# The code / scale rule and the padding check (tests/acceptance.py), on the
# oracle's own output with planted differences.
# ---------------------------------------------------------------------------
import acceptance  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402


def _oracle_case(M, H, fmt, layout="swizzled", seed=0):
    wl = workloads.Workload("t", M, H, "bf16", fmt, layout, 1e-6, seed=seed)
    x, r, w = workloads.make_inputs(wl, "cpu")
    o = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                     wl.eps, "bf16", fmt, layout)
    return x, r, w, o


@pytest.mark.parametrize("M,H,fmt", [(1, 64, "nvfp4"), (130, 80, "nvfp4"), (129, 96, "mxfp4"),
                                     (256, 256, "nvfp4"), (5, 224, "e4m3b32")])
def test_tiled_padding_check(M, H, fmt):
    """The oracle's tiled buffer passes; a nonzero byte in any padding slot
    (rows past M, or k past nb) fails; data bytes may hold anything."""
    _, _, _, o = _oracle_case(M, H, fmt)
    nb = H // oracle.block_size(fmt)
    sf = o.sf_swizzled.copy()
    assert acceptance.tiled_padding_is_zero(sf, M, nb)
    nkt = (nb + 3) // 4
    data = np.zeros(sf.size, bool)
    mm, kk = np.meshgrid(np.arange(M), np.arange(nb), indexing="ij")
    data[oracle.swizzled_sf_offset(mm, kk, nkt).reshape(-1)] = True
    sf2 = sf.copy()
    sf2[data] = 0x5A
    assert acceptance.tiled_padding_is_zero(sf2, M, nb)
    for i in np.flatnonzero(~data)[:50]:
        sf3 = sf.copy()
        sf3[i] = 1
        assert not acceptance.tiled_padding_is_zero(sf3, M, nb), i


def test_check_rows_accepts_the_oracle_and_rejects_planted_flips():
    x, r, w, o = _oracle_case(8, 256, "nvfp4", "rowmajor", seed=3)
    res = acceptance.residual_bits(o.residual, "bf16")
    assert acceptance.check_rows(o, res, o.scale_codes, o.packed, "nvfp4", "bf16") == 0
    # a code flipped where v is far from an E2M1 midpoint
    far = np.argwhere(~acceptance.near(np.abs(o.v), acceptance.E2M1_MIDS))[0]
    pk = o.packed.copy()
    j = far[1] // 2
    pk[far[0], j] ^= 0x01 if far[1] % 2 == 0 else 0x10
    with pytest.raises(AssertionError, match="codes differ"):
        acceptance.check_rows(o, res, o.scale_codes, pk, "nvfp4", "bf16")
    # a scale byte changed away from an E4M3 midpoint
    sc = o.scale_codes.copy()
    sc[0, 0] ^= 0x01
    with pytest.raises(AssertionError, match="scale bytes differ"):
        acceptance.check_rows(o, res, sc, o.packed, "nvfp4", "bf16")
    # one residual bit
    res2 = res.copy()
    res2[1, 7] ^= 1
    with pytest.raises(AssertionError, match="residual differs"):
        acceptance.check_rows(o, res2, o.scale_codes, o.packed, "nvfp4", "bf16")


def test_block_task_matches_whole_batch():
    """The worker task on row blocks counts what the whole-batch rule counts
    and reads the 16-bit inputs back exactly."""
    x, r, w, o = _oracle_case(40, 512, "mxfp4", "rowmajor", seed=5)
    xb = x.view(torch_int16()).numpy().view(np.uint16)
    rb = r.view(torch_int16()).numpy().view(np.uint16)
    res = acceptance.residual_bits(o.residual, "bf16")
    tot = 0
    for a in range(0, 40, 16):
        b = min(40, a + 16)
        n, e = acceptance.fused_block_task((xb[a:b], rb[a:b], w.float().numpy(), 1e-6, "bf16",
                                            "mxfp4", res[a:b], o.packed[a:b],
                                            o.scale_codes[a:b]))
        assert n == 0 and e == (b - a) * 512
        tot += e
    assert tot == o.codes.size


def torch_int16():
    import torch
    return torch.int16
