"""Pins for the oracle's number formats, against things other than itself:
exhaustive tables written from the format definitions, torch's CPU casts
(library routines) and brute-force nearest-value search."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F

# E2M1: sign bit, two exponent bits (bias 1), one mantissa bit; exponent 0 is
# subnormal (0 or 0.5).  Written out by hand from that definition.
E2M1_TABLE = {
    0x0: 0.0, 0x1: 0.5, 0x2: 1.0, 0x3: 1.5, 0x4: 2.0, 0x5: 3.0, 0x6: 4.0, 0x7: 6.0,
    0x8: -0.0, 0x9: -0.5, 0xA: -1.0, 0xB: -1.5, 0xC: -2.0, 0xD: -3.0, 0xE: -4.0, 0xF: -6.0,
}


def test_e2m1_decode_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    got = oracle.e2m1_decode(codes)
    for c in range(16):
        assert got[c] == E2M1_TABLE[c]
        assert np.signbit(got[c]) == (c >= 8) or E2M1_TABLE[c] != 0


def test_e2m1_encode_inverts_decode():
    for c in range(16):
        v = np.float32(E2M1_TABLE[c])
        if c == 0x8:
            v = np.float32(-0.0)
        assert int(oracle.e2m1_encode(np.array([v]))[0]) == c


def _brute_e2m1(v):
    """Nearest of the 16 codes by exhaustive search in fp64; ties between two
    magnitudes go to the even mantissa bit, ties between +0/-0 to the sign of v."""
    vals = np.array([E2M1_TABLE[c] for c in range(16)], dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        clamped = np.clip(x, -6.0, 6.0)
        d = np.abs(vals - clamped)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            mags = {c & 7 for c in best}
            if len(mags) > 1:                       # tie between two magnitudes
                best = [c for c in best if (c & 1) == 0]
            if len(best) > 1:                       # +0 / -0
                want_neg = bool(np.signbit(x))
                best = [c for c in best if (c >= 8) == want_neg]
        assert len(best) == 1, (x, best)
        out[i] = best[0]
    return out


def test_e2m1_encode_matches_brute_force():
    rng = np.random.default_rng(0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    around = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                             np.nextafter(mids, np.float32(10))])
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, 6.5, 7, 100, 1e30], dtype=np.float32)
    rand = rng.uniform(-7, 7, 20000).astype(np.float32)
    tiny = np.array([1e-30, 1e-45, 0.1, 0.2499999], dtype=np.float32)
    v = np.concatenate([around, -around, grid, -grid, rand, tiny, -tiny,
                        np.array([0.0, -0.0], np.float32)])
    assert np.array_equal(oracle.e2m1_encode(v), _brute_e2m1(v))


def test_e2m1_ties_go_to_even():
    # the seven midpoints and where they must land
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for m, want in expect.items():
        got = oracle.e2m1_decode(oracle.e2m1_encode(np.array([m], np.float32)))[0]
        assert got == want, (m, got)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    finite = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float32)
    mids = ((finite[:-1].astype(np.float64) + finite[1:]) / 2).astype(np.float32)
    edges = np.concatenate([finite, mids, np.nextafter(mids, np.float32(0)),
                            np.nextafter(mids, np.float32(1000))])
    # log-uniform over the whole range including subnormals
    rand = np.exp2(rng.uniform(-12, np.log2(448), 1_000_000)).astype(np.float32)
    t = np.concatenate([edges, rand, np.array([0.0, 448.0, 2.0 ** -10, 1e-30], np.float32)])
    t = t[(t >= 0) & (t <= 448)]
    ours = oracle.e4m3_encode_rne(t)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, (t[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(2)
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    t = np.exp2(rng.uniform(-11, 8.8, 5000)).astype(np.float32)
    t = t[t <= 448]
    codes = oracle.e4m3_encode_rne(t)
    for ti, c in zip(t.astype(np.float64), codes):
        d = np.abs(vals - ti)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if b % 2 == 0]
        assert c == best[0]


def test_ue8m0_exhaustive_and_ceiling():
    codes = np.arange(255, dtype=np.uint8)
    dec = oracle.ue8m0_decode(codes)
    assert np.all(dec.astype(np.float64) == np.exp2(codes.astype(np.float64) - 127))
    assert np.isnan(oracle.ue8m0_decode(np.array([255], np.uint8))[0])
    for e in range(-126, 128):
        p = np.float32(2.0 ** e)
        assert oracle.ue8m0_encode_ceil(np.array([p]))[0] == e + 127
        above = np.nextafter(p, np.float32(np.inf))
        if e < 127:
            assert oracle.ue8m0_encode_ceil(np.array([above]))[0] == e + 128
        below = np.nextafter(p, np.float32(0))
        assert oracle.ue8m0_encode_ceil(np.array([below]))[0] == e + 127
    # subnormal fp32 and zero
    assert oracle.ue8m0_encode_ceil(np.array([2.0 ** -127], np.float32))[0] == 0
    assert oracle.ue8m0_encode_ceil(np.array([2.0 ** -130], np.float32))[0] == 0
    assert oracle.ue8m0_encode_ceil(np.array([0.0], np.float32))[0] == 0
    assert oracle.ue8m0_encode_ceil(np.array([1.5 * 2.0 ** -127], np.float32))[0] == 1


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_dtype_rounding_matches_torch(dtype, tdt):
    rng = np.random.default_rng(3)
    a = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 10,
                        (1 + np.arange(-2000, 2000) * 2.0 ** -17).astype(np.float32)])
    ours = oracle.round_to_dtype(a, dtype)
    ref = torch.from_numpy(a).to(tdt).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_bf16_tie_cases():
    assert F.bf16_round(np.array([1 + 2.0 ** -8], np.float32))[0] == 1.0
    assert F.bf16_round(np.array([1 + 3 * 2.0 ** -8], np.float32))[0] == 1 + 2.0 ** -6
