"""Pins of the consumer-GEMM oracle (``oracle.gemm``) against closed forms,
brute force and the quantization error bound.  CPU only.

Inputs are built from explicit codes and scale bytes; the decoding of a code
or a scale byte is pinned by the format tests, the tiled offset by the
nested-tile test, so what is pinned here is the contraction itself: which
operand is transposed, which scale buffer goes with which operand, alpha,
the epilogue terms and the final rounding.
"""
import inspect

import numpy as np
import pytest

import oracle
from oracle import gemm as OG

E4M3_ONE, E4M3_TWO, E4M3_HALF, E4M3_QUARTER, E4M3_FOUR = 0x38, 0x40, 0x30, 0x28, 0x48
E2M1_ONE, E2M1_TWO, E2M1_HALF = 0x2, 0x4, 0x1


def pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def tiled(scale_codes):
    """Scale bytes (rows, nb) into a zeroed 128x4 tiled buffer."""
    sc = np.asarray(scale_codes, np.uint8)
    R, nb = sc.shape
    buf = np.zeros(oracle.sf_size_bytes(R, nb * 16, "nvfp4", "swizzled"), np.uint8)
    mm, kk = np.meshgrid(np.arange(R), np.arange(nb), indexing="ij")
    buf[oracle.swizzled_sf_offset(mm, kk, (nb + 3) // 4)] = sc
    return buf


def run(a_codes, a_sc, b_codes, b_sc, alpha=1.0, bias=None, residual=None):
    M, K = a_codes.shape
    N = b_codes.shape[0]
    return oracle.gemm_bf16(pack(a_codes), pack(b_codes), tiled(a_sc), tiled(b_sc), M, N, K,
                            alpha=alpha, bias=bias, residual=residual)


def test_constant_operands_closed_form():
    M, N, K = 3, 5, 128
    a = np.full((M, K), E2M1_ONE, np.uint8)
    b = np.full((N, K), E2M1_TWO, np.uint8)
    g = run(a, np.full((M, K // 16), E4M3_ONE), b, np.full((N, K // 16), E4M3_HALF), alpha=0.25)
    assert np.all(g.exact == K * 1.0 * 2.0 * 0.5 * 0.25)
    assert np.all(g.out == K / 4)
    assert np.all(g.bound == K / 4)


def test_one_hot_rows_select_a_row_of_b():
    """A row m holds a single 1.0 at k = 3m + 1: out[m, n] = deq(B)[n, 3m + 1],
    which fails for B not transposed or for the scale buffers swapped."""
    rng = np.random.default_rng(1)
    M, N, K = 4, 6, 64
    a = np.zeros((M, K), np.uint8)
    for m in range(M):
        a[m, 3 * m + 1] = E2M1_ONE
    b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    b_sc = rng.choice([E4M3_HALF, E4M3_ONE, E4M3_TWO, E4M3_FOUR], (N, K // 16))
    g = run(a, np.full((M, K // 16), E4M3_ONE), b, b_sc)
    deq_b = oracle.dequant(pack(b), tiled(b_sc), N, K, "nvfp4", "swizzled")
    for m in range(M):
        assert np.array_equal(g.exact[m], deq_b[:, 3 * m + 1].astype(np.float64))


def test_row_and_block_scales_multiply():
    """Per-row scales of A and of B and per-block scales along k: out[m, n] =
    sum over blocks of 16 * sa[m, blk] * sb[n, blk]."""
    M, N, K = 5, 3, 64
    pw = {0: E4M3_ONE, 1: E4M3_TWO, 2: E4M3_FOUR, -1: E4M3_HALF, -2: E4M3_QUARTER}
    ea = np.array([[(m % 3) - 1 + (k % 2) for k in range(K // 16)] for m in range(M)])
    eb = np.array([[-(n % 2) - (k // 2) for k in range(K // 16)] for n in range(N)])
    a_sc = np.vectorize(pw.get)(ea)
    b_sc = np.vectorize(pw.get)(eb)
    g = run(np.full((M, K), E2M1_ONE, np.uint8), a_sc, np.full((N, K), E2M1_ONE, np.uint8), b_sc)
    want = np.array([[sum(16 * 2.0 ** (ea[m, k] + eb[n, k]) for k in range(K // 16))
                      for n in range(N)] for m in range(M)])
    assert np.array_equal(g.exact, want)


def test_bias_and_residual_added_after_alpha():
    M, N, K = 2, 4, 32
    a = np.full((M, K), E2M1_ONE, np.uint8)
    b = np.full((N, K), E2M1_ONE, np.uint8)
    one = np.full((M, K // 16), E4M3_ONE)
    bias = np.array([1.0, -2.0, 3.0, 0.5], np.float32)
    res = np.arange(M * N, dtype=np.float32).reshape(M, N)
    g = run(a, one, b, np.full((N, K // 16), E4M3_ONE), alpha=0.5, bias=bias, residual=res)
    assert np.array_equal(g.exact, K * 0.5 + bias[None, :] + res)
    assert np.array_equal(g.out, (K * 0.5 + bias[None, :] + res).astype(np.float32))


def test_output_rounds_to_nearest_even_bf16():
    """1 + 2^-8 is a bf16 tie (to 1.0); 1 + 2^-8 + 2^-10 rounds up to 1 + 2^-7."""
    K = 48
    a = np.zeros((2, K), np.uint8)
    a[:, 0] = E2M1_ONE           # block 0, scale 1.0: 1.0
    a[:, 16] = E2M1_ONE          # block 1, scale 2^-8 (E4M3 subnormal 0x02): 2^-8
    a[1, 32] = E2M1_HALF         # block 2, scale 2^-9 (0x01): 0.5 * 2^-9 = 2^-10
    a_sc = np.array([[E4M3_ONE, 0x02, 0x01]] * 2)
    g = run(a, a_sc, np.full((1, K), E2M1_ONE, np.uint8), np.full((1, K // 16), E4M3_ONE))
    assert g.exact[0, 0] == 1 + 2.0 ** -8 and g.out[0, 0] == 1.0
    assert g.exact[1, 0] == 1 + 2.0 ** -8 + 2.0 ** -10 and g.out[1, 0] == 1 + 2.0 ** -7


def _e2m1(c):
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0][c & 7]
    return -mag if c & 8 else mag


def _e4m3(byte):
    e, m = (byte >> 3) & 15, byte & 7
    return (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)


def test_brute_force_tiny():
    """Element by element from the codes and scale bytes, the sum over k in
    Python floats, against the oracle's matrix product."""
    rng = np.random.default_rng(7)
    M, N, K = 3, 5, 32
    a = rng.integers(0, 16, (M, K)).astype(np.uint8)
    b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    a_sc = rng.integers(0x20, 0x50, (M, K // 16))
    b_sc = rng.integers(0x20, 0x50, (N, K // 16))
    g = run(a, a_sc, b, b_sc, alpha=1.5)
    for m in range(M):
        for n in range(N):
            s = sum(_e2m1(a[m, k]) * _e4m3(a_sc[m, k // 16]) * _e2m1(b[n, k]) * _e4m3(b_sc[n, k // 16])
                    for k in range(K))
            assert g.exact[m, n] == pytest.approx(1.5 * s, rel=1e-14, abs=1e-300)


UE8M0_ONE = 127


def tiled_mx(scale_codes):
    """UE8M0 scale bytes (rows, nb) into a zeroed 128x4 tiled buffer (32-blocks)."""
    sc = np.asarray(scale_codes, np.uint8)
    R, nb = sc.shape
    buf = np.zeros(oracle.sf_size_bytes(R, nb * 32, "mxfp4", "swizzled"), np.uint8)
    mm, kk = np.meshgrid(np.arange(R), np.arange(nb), indexing="ij")
    buf[oracle.swizzled_sf_offset(mm, kk, (nb + 3) // 4)] = sc
    return buf


def test_mxfp4_row_and_block_scales_multiply():
    """MXFP4 operands (UE8M0 scale per 32 codes): per-row and per-block powers
    of two multiply as in the NVFP4 case, 32 elements per block."""
    M, N, K = 3, 5, 128
    ea = np.array([[(m % 3) - 1 + (k % 2) for k in range(K // 32)] for m in range(M)])
    eb = np.array([[-(n % 2) - (k // 2) + 2 for k in range(K // 32)] for n in range(N)])
    a = np.full((M, K), E2M1_ONE, np.uint8)
    b = np.full((N, K), E2M1_TWO, np.uint8)
    g = oracle.gemm_bf16(pack(a), pack(b), tiled_mx(UE8M0_ONE + ea), tiled_mx(UE8M0_ONE + eb),
                         M, N, K, fmt="mxfp4")
    want = np.array([[sum(32 * 2.0 * 2.0 ** (ea[m, k] + eb[n, k]) for k in range(K // 32))
                      for n in range(N)] for m in range(M)])
    assert np.array_equal(g.exact, want)


def test_mxfp4_brute_force_tiny():
    rng = np.random.default_rng(9)
    M, N, K = 2, 3, 64
    a = rng.integers(0, 16, (M, K)).astype(np.uint8)
    b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    a_sc = rng.integers(120, 135, (M, K // 32))
    b_sc = rng.integers(120, 135, (N, K // 32))
    g = oracle.gemm_bf16(pack(a), pack(b), tiled_mx(a_sc), tiled_mx(b_sc), M, N, K, alpha=0.5,
                         fmt="mxfp4")
    for m in range(M):
        for n in range(N):
            s = sum(_e2m1(a[m, k]) * 2.0 ** (int(a_sc[m, k // 32]) - 127) *
                    _e2m1(b[n, k]) * 2.0 ** (int(b_sc[n, k // 32]) - 127) for k in range(K))
            assert g.exact[m, n] == pytest.approx(0.5 * s, rel=1e-14, abs=1e-300)


def test_quantized_product_within_quantization_bound():
    """x and w quantized by the producer oracle, then multiplied: the result
    is x @ w^T up to the per-element quantization errors, each at most one
    block scale (half the widest E2M1 step), weighted by the other operand."""
    rng = np.random.default_rng(3)
    M, N, K = 8, 16, 256
    x = oracle.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    w = oracle.bf16_round(rng.standard_normal((N, K)).astype(np.float32))
    qx = oracle.quantize(x, "nvfp4", "swizzled")
    qw = oracle.quantize(w, "nvfp4", "swizzled")
    g = oracle.gemm_bf16(qx.packed, qw.packed, qx.sf_swizzled, qw.sf_swizzled, M, N, K)
    dx = oracle.dequant(qx.packed, qx.sf_swizzled, M, K, "nvfp4", "swizzled").astype(np.float64)
    dw = oracle.dequant(qw.packed, qw.sf_swizzled, N, K, "nvfp4", "swizzled").astype(np.float64)
    sx = np.repeat(oracle.e4m3_decode(qx.scale_codes), 16, axis=1).astype(np.float64)
    sw = np.repeat(oracle.e4m3_decode(qw.scale_codes), 16, axis=1).astype(np.float64)
    bound = sx @ np.abs(dw).T + np.abs(x) @ sw.T
    err = np.abs(g.exact - x.astype(np.float64) @ w.astype(np.float64).T)
    assert np.all(err <= bound * (1 + 1e-12))
    assert np.all(err <= 0.5 * np.abs(x) @ np.abs(w).T)   # and not vacuous


# ---------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin above
# ---------------------------------------------------------------------------
GEMM_MUTANTS = {
    "B not transposed": ("s = a @ b.T", "s = a @ b"),
    "scale buffers swapped": ("a = dequant(a_packed, sfa,", "a = dequant(a_packed, sfb,"),
    "alpha dropped": ("exact = alpha64 * s", "exact = s"),
    "bias scaled by alpha": ("exact = exact + np.asarray(bias, np.float64).reshape(1, N)",
                             "exact = exact + alpha64 * np.asarray(bias, np.float64).reshape(1, N)"),
    "residual ignored": ("exact = exact + np.asarray(residual, np.float64).reshape(M, N)",
                         "exact = exact"),
    "output truncated": ("out = bf16_round(exact.astype(np.float32))",
                         "out = ((exact.astype(np.float32).view(np.uint32) >> 16) << 16)"
                         ".astype(np.uint32).view(np.float32)"),
}

PINS = [test_constant_operands_closed_form, test_one_hot_rows_select_a_row_of_b,
        test_row_and_block_scales_multiply, test_bias_and_residual_added_after_alpha,
        test_output_rounds_to_nearest_even_bf16, test_brute_force_tiny,
        test_quantized_product_within_quantization_bound]


@pytest.mark.parametrize("name", list(GEMM_MUTANTS))
def test_gemm_mutant_is_caught(name, monkeypatch):
    old, new = GEMM_MUTANTS[name]
    src = inspect.getsource(OG.gemm_bf16)
    assert old in src, f"mutation anchor not found: {old!r}"
    ns = dict(vars(OG))
    exec(compile(src.replace(old, new, 1), "<mutant gemm_bf16>", "exec"), ns)
    monkeypatch.setattr(oracle, "gemm_bf16", ns["gemm_bf16"])
    caught = False
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, f"no pin caught: {name}"


# ---------------------------------------------------------------------------
# GELU epilogues
# ---------------------------------------------------------------------------
# standard normal CDF at 0.5, 1, 2 (printed tables of Phi)
PHI = {0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 2.0: 0.9772498680518208}


def test_gelu_is_x_times_normal_cdf():
    for x, phi in PHI.items():
        assert oracle.gelu(x) == pytest.approx(x * phi, rel=1e-15)
        # Phi(-x) = 1 - Phi(x)
        assert oracle.gelu(-x) == pytest.approx(-x * (1 - phi), rel=1e-14)
    assert oracle.gelu(0.0) == 0.0
    xs = np.linspace(-6, 6, 97)
    assert np.allclose(oracle.gelu(xs) - oracle.gelu(-xs), xs, rtol=0, atol=1e-15)


def test_gemm_gelu_applies_to_alpha_product_plus_bias():
    """One-hot rows select a column of deq(B): out = GELU(alpha * b + bias)."""
    rng = np.random.default_rng(4)
    M, N, K = 3, 8, 64
    a = np.zeros((M, K), np.uint8)
    for m in range(M):
        a[m, 5 * m] = E2M1_ONE
    b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    b_sc = np.full((N, K // 16), E4M3_ONE)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    g = oracle.gemm_bf16(pack(a), pack(b), tiled(np.full((M, K // 16), E4M3_ONE)), tiled(b_sc),
                         M, N, K, alpha=0.5, bias=bias, gelu_act=True)
    deq_b = oracle.dequant(pack(b), tiled(b_sc), N, K, "nvfp4", "swizzled").astype(np.float64)
    for m in range(M):
        x = 0.5 * deq_b[:, 5 * m] + bias
        assert np.allclose(g.exact[m], x * 0.5 * (1 + np.vectorize(__import__("math").erf)(
            x / np.sqrt(2))), rtol=1e-14, atol=1e-300)
    with pytest.raises(ValueError):
        oracle.gemm_bf16(pack(a), pack(b), tiled(np.full((M, K // 16), E4M3_ONE)), tiled(b_sc),
                         M, N, K, residual=np.zeros((M, N)), gelu_act=True)


def test_gemm_gelu_nvfp4_output_dequantises_near_gelu():
    """The FP4-output epilogue: every code, times its block scale, is within
    half an E2M1 step (times the scale) of the GELU value it encodes."""
    rng = np.random.default_rng(6)
    M, N, K = 5, 64, 128
    a = rng.integers(0, 16, (M, K)).astype(np.uint8)
    b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    a_sc = rng.integers(0x30, 0x40, (M, K // 16))
    b_sc = rng.integers(0x30, 0x40, (N, K // 16))
    bias = rng.standard_normal(N).astype(np.float32)
    q = oracle.gemm_gelu_nvfp4(pack(a), pack(b), tiled(a_sc), tiled(b_sc), M, N, K, alpha=0.25,
                               bias=bias)
    g = oracle.gemm_bf16(pack(a), pack(b), tiled(a_sc), tiled(b_sc), M, N, K, alpha=0.25,
                         bias=bias, gelu_act=True)
    deq = oracle.dequant(q.packed, q.sf_swizzled, M, N, "nvfp4", "swizzled").astype(np.float64)
    s = np.repeat(oracle.e4m3_decode(q.scale_codes), 16, axis=1).astype(np.float64)
    v = g.exact / np.where(s > 0, s, 1)
    step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0))
    err = np.abs(deq - g.exact)
    assert np.all(err <= np.maximum(0.5 * step * s * (1 + 1e-6), (np.abs(v) - 6) * s + 1e-12))


GELU_MUTANTS = {
    "tanh approximation": ("return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))",
                           "return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * "
                           "(x + 0.044715 * x ** 3)))"),
    "erf argument not scaled": ("erf(x / np.sqrt(2.0))", "erf(x)"),
    "Phi instead of x * Phi": ("return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))",
                               "return 0.5 * (1.0 + erf(x / np.sqrt(2.0)))"),
}


@pytest.mark.parametrize("name", list(GELU_MUTANTS))
def test_gelu_mutant_is_caught(name, monkeypatch):
    old, new = GELU_MUTANTS[name]
    src = inspect.getsource(OG.gelu)
    assert old in src
    ns = dict(vars(OG))
    exec(compile(src.replace(old, new, 1), "<mutant gelu>", "exec"), ns)
    monkeypatch.setattr(oracle, "gelu", ns["gelu"])
    monkeypatch.setattr(OG, "gelu", ns["gelu"])
    with pytest.raises(AssertionError):
        test_gelu_is_x_times_normal_cdf()
