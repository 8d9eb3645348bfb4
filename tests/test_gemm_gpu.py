"""GPU parity of the NVFP4 GEMM (fp4_gemm_nvfp4_bf16, through the C ABI via the
binding) against the oracle (``oracle.gemm_bf16``).

Two kinds of operands, both drawn as bytes by ``workloads.random_bytes``:
  * "exact": codes in {0, +-0.5, +-1, +-2} and scales in {0.5, 1, 2}.  Every
    product is a multiple of 2^-4 of magnitude <= 16 and every partial sum
    stays below 2^17 for K <= 7168, so any fp32 summation order is exact and
    the bf16 output must equal the oracle's bit for bit;
  * "random": every E2M1 code, scales 2^-3 .. 9.  The tensor cores sum in fp32
    in their own order, so the output must lie within
        2^-8 |exact| + 2^-22 K sum_k |a b| + 2^-22 (|bias| + |residual|)
    of the oracle's exact value: one bf16 rounding (2^-9, doubled), K fp32
    additions each off by at most 2^-23 relative to the running magnitude
    (doubled), and one rounding per epilogue addition.
"""
import numpy as np
import pytest
import torch

import acceptance
import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads

pytestmark = pytest.mark.gpu

E2M1_SMALL = [0x0, 0x1, 0x2, 0x4, 0x9, 0xA, 0xC]      # 0, +-0.5, +-1, +-2
EXACT_BYTES = [lo | (hi << 4) for lo in E2M1_SMALL for hi in E2M1_SMALL]
# scale bytes per format: powers of two 0.5, 1, 2 (exact kind) and a range
SCALES = {"nvfp4": {"exact": [0x30, 0x38, 0x40], "random": list(range(0x20, 0x51))},   # 2^-3..9
          "mxfp4": {"exact": [126, 127, 128], "random": list(range(122, 133))}}       # 2^-5..2^5


def operands(M, N, K, seed, kind, fmt="nvfp4"):
    code_alpha = EXACT_BYTES if kind == "exact" else None
    sf_alpha = SCALES[fmt][kind]
    a = workloads.random_bytes(M * K // 2, seed, 0, code_alpha).reshape(M, K // 2)
    b = workloads.random_bytes(N * K // 2, seed, 1, code_alpha).reshape(N, K // 2)
    sfa = workloads.random_bytes(oracle.sf_size_bytes(M, K, fmt, "swizzled"), seed, 2, sf_alpha)
    sfb = workloads.random_bytes(oracle.sf_size_bytes(N, K, fmt, "swizzled"), seed, 3, sf_alpha)
    return a, b, sfa, sfb


def bf16_values(n, seed, tensor_id, shape):
    """bf16 tensors whose values are multiples of 2^-4 below 2^9 in magnitude
    (exact in every fp32 sum of the exact-kind tests)."""
    ints = workloads.random_bytes(n, seed, tensor_id).to(torch.int32) - 128
    return (ints.to(torch.float32) * 0.25).to(torch.bfloat16).reshape(shape)


def gpu_gemm(a, b, sfa, sfb, alpha=1.0, bias=None, residual=None, out=None, pdl=False,
             variant=-1, fmt="nvfp4"):
    dev = "cuda"
    res = fq.gemm_nvfp4_bf16(a.to(dev), b.to(dev), sfa.to(dev), sfb.to(dev), alpha=alpha,
                             bias=None if bias is None else bias.to(dev),
                             residual=residual, out=out, pdl=pdl, variant=variant, fmt=fmt)
    torch.cuda.synchronize()
    return res


def check(got, g, K, kind, bias=None, residual=None):
    got64 = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got64).all(), "non-finite output (a bounded wait ran out?)"
    if kind == "exact":
        bad = got64.astype(np.float32) != g.out
        assert not bad.any(), (f"{bad.sum()} outputs differ, first at {np.argwhere(bad)[:4].tolist()}: "
                               f"gpu {got64[bad][:4]} oracle {g.out[bad][:4]}")
        return
    tol = 2.0 ** -8 * np.abs(g.exact) + 2.0 ** -22 * K * g.bound
    if bias is not None:
        tol = tol + 2.0 ** -22 * np.abs(bias.float().numpy().astype(np.float64))[None, :]
    if residual is not None:
        tol = tol + 2.0 ** -22 * np.abs(residual.float().cpu().numpy().astype(np.float64))
    err = np.abs(got64 - g.exact)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} outputs outside the bound, first at "
                           f"{np.argwhere(bad)[:4].tolist()}: gpu {got64[bad][:4]} "
                           f"exact {g.exact[bad][:4]} tol {tol[bad][:4]}")


def oracle_gemm(a, b, sfa, sfb, M, N, K, **kw):
    return oracle.gemm_bf16(a.numpy(), b.numpy(), sfa.numpy(), sfb.numpy(), M, N, K, **kw)


EXACT_SHAPES = [(128, 128, 256), (1, 8, 256), (41, 4608, 1536), (300, 520, 768),
                (129, 136, 512), (256, 1024, 4096)]

MX_VARIANTS = [0, 1, 2, 3, 4]   # MXFP4: every schedule, as for NVFP4


@pytest.mark.parametrize("M,N,K", EXACT_SHAPES)
@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_gemm_mxfp4_exact_operands_bit_exact(M, N, K, variant):
    """MXFP4 operands (UE8M0 per 32 codes; two 128x4 scale tiles per K block,
    each holding two K steps' scales)."""
    a, b, sfa, sfb = operands(M, N, K, seed=7 * M + N + K, kind="exact", fmt="mxfp4")
    got = gpu_gemm(a, b, sfa, sfb, alpha=0.5, variant=variant, fmt="mxfp4")
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.5, fmt="mxfp4"), K, "exact")


@pytest.mark.parametrize("M,N,K", [(256, 384, 2048), (41, 1536, 6144)])
@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_gemm_mxfp4_random_operands(M, N, K, variant):
    a, b, sfa, sfb = operands(M, N, K, seed=5 * M + N, kind="random", fmt="mxfp4")
    got = gpu_gemm(a, b, sfa, sfb, variant=variant, fmt="mxfp4")
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, fmt="mxfp4"), K, "random")


VARIANTS = [0, 1, 2, 3, 4]   # 128x128 / 128x256 tiles; one CTA per tile / persistent; split K


@pytest.mark.parametrize("M,N,K", EXACT_SHAPES)
@pytest.mark.parametrize("alpha", [1.0, 0.5])
@pytest.mark.parametrize("variant", VARIANTS)
def test_gemm_exact_operands_bit_exact(M, N, K, alpha, variant):
    """One tile, the minimal shape, a release-gate shape, ragged M and N tails
    (a partial last row tile and an 8-column last column tile; with 256-wide
    tiles a last tile holding one 128-row scale tile of B), many K blocks."""
    a, b, sfa, sfb = operands(M, N, K, seed=M + N + K, kind="exact")
    got = gpu_gemm(a, b, sfa, sfb, alpha=alpha, variant=variant)
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=alpha), K, "exact")


# Split K (variant 4) reduces through the ranks' shared memory: each rank owns
# rows [q * rows / split, (q + 1) * rows / split) of the tile and receives
# those rows of every other rank's partial.  Shapes where most ranks own no row
# (1 or 5 rows over 16 ranks), a full 128-row tile over 16 ranks (the receive
# slots then need a deeper ring than the default), and a ragged K.
SPLIT_SHAPES = [(1, 8, 4096), (5, 264, 4096), (128, 128, 8192), (41, 1536, 6144),
                (130, 264, 4000)]


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_gemm_split_k_reduction_bit_exact(M, N, K, fmt):
    a, b, sfa, sfb = operands(M, N, K, seed=M + 7 * N + K, kind="exact", fmt=fmt)
    assert fq.fp4_gemm_variant(M, N, K, fmt=0 if fmt == "nvfp4" else 1, variant=4)["split_k"]
    got = gpu_gemm(a, b, sfa, sfb, alpha=0.5, variant=4, fmt=fmt)
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.5, fmt=fmt), K, "exact")


@pytest.mark.parametrize("M,N,K,variant", [(41, 1536, 6144, 4), (130, 264, 4000, 4),
                                           (41, 4608, 1536, 0), (256, 768, 2048, 3)])
def test_gemm_repeats_bit_identical(M, N, K, variant):
    """The split-K reduction sums the ranks in a fixed order and the epilogues
    write each output once, so repeated launches give identical bytes."""
    a, b, sfa, sfb = operands(M, N, K, seed=M * 3 + N + K, kind="random")
    dev = [t.cuda() for t in (a, b, sfa, sfb)]
    first = fq.gemm_nvfp4_bf16(*dev, alpha=0.5, variant=variant)
    outs = [fq.gemm_nvfp4_bf16(*dev, alpha=0.5, variant=variant) for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), first.view(torch.int16))


# K not a multiple of 256: a ragged last K block of 1-4 K = 64 steps, the last
# of them possibly half past K (codes there read as zero, scales are the
# k-padding of the tiled layout)
RAGGED_K_SHAPES = [(128, 128, 32), (1, 8, 96), (128, 128, 224), (41, 520, 288),
                   (77, 264, 352), (300, 136, 800), (129, 264, 1600), (256, 384, 4160)]


@pytest.mark.parametrize("M,N,K", RAGGED_K_SHAPES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_gemm_ragged_k_bit_exact(M, N, K, variant):
    a, b, sfa, sfb = operands(M, N, K, seed=3 * M + N + K, kind="exact")
    got = gpu_gemm(a, b, sfa, sfb, alpha=0.5, variant=variant)
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.5), K, "exact")


@pytest.mark.parametrize("M,N,K", RAGGED_K_SHAPES)
@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_gemm_mxfp4_ragged_k_bit_exact(M, N, K, variant):
    a, b, sfa, sfb = operands(M, N, K, seed=5 * M + N + K, kind="exact", fmt="mxfp4")
    got = gpu_gemm(a, b, sfa, sfb, variant=variant, fmt="mxfp4")
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, fmt="mxfp4"), K, "exact")


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_gemm_ragged_k_random_operands(fmt):
    M, N, K = 200, 392, 2144          # 8 full K blocks and one of 96 codes
    a, b, sfa, sfb = operands(M, N, K, seed=11, kind="random", fmt=fmt)
    got = gpu_gemm(a, b, sfa, sfb, alpha=1.25, fmt=fmt)
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=1.25, fmt=fmt), K, "random")


def test_gemm_rejects_k_not_multiple_of_32():
    """K = 240 is a whole number of NVFP4 blocks, but a row of 120 bytes is no
    multiple of 16 bytes, which the tiled loads need."""
    a, b, sfa, sfb = operands(128, 128, 240, 1, "exact")
    with pytest.raises(fq.Fp4Error):
        gpu_gemm(a, b, sfa, sfb)


@pytest.mark.parametrize("name", ["G1_M41_N4608_K1536", "G2_M41_N6144_K1536",
                                  "G3_M41_N1536_K6144"])
def test_gemm_release_gate_shapes_random_operands(name):
    wl = workloads.GEMM_CONFIGS[name]
    a, b, sfa, sfb = operands(wl.M, wl.N, wl.K, wl.seed, "random")
    got = gpu_gemm(a, b, sfa, sfb, alpha=0.75)
    check(got, oracle_gemm(a, b, sfa, sfb, wl.M, wl.N, wl.K, alpha=0.75), wl.K, "random")


@pytest.mark.parametrize("M,N,K", [(256, 384, 2048), (77, 264, 512)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_gemm_random_operands(M, N, K, variant):
    a, b, sfa, sfb = operands(M, N, K, seed=3 * M + N, kind="random")
    got = gpu_gemm(a, b, sfa, sfb, variant=variant)
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K), K, "random")


@pytest.mark.parametrize("with_bias,with_residual", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_gemm_bias_residual_epilogues(with_bias, with_residual, variant):
    M, N, K = 200, 264, 1024
    a, b, sfa, sfb = operands(M, N, K, seed=21, kind="exact")
    bias = bf16_values(N, 21, 4, (N,)) if with_bias else None
    res = bf16_values(M * N, 21, 5, (M, N)) if with_residual else None
    got = gpu_gemm(a, b, sfa, sfb, alpha=0.5, bias=bias,
                   residual=None if res is None else res.cuda(), variant=variant)
    g = oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.5,
                    bias=None if bias is None else bias.float().numpy(),
                    residual=None if res is None else res.float().numpy())
    check(got, g, K, "exact")


def test_gemm_residual_in_place():
    """residual == out: each element read, then overwritten, by one thread."""
    M, N, K = 130, 256, 512
    a, b, sfa, sfb = operands(M, N, K, seed=22, kind="exact")
    res = bf16_values(M * N, 22, 5, (M, N))
    buf = res.cuda()
    got = gpu_gemm(a, b, sfa, sfb, residual=buf, out=buf)
    assert got.data_ptr() == buf.data_ptr()
    check(got, oracle_gemm(a, b, sfa, sfb, M, N, K, residual=res.float().numpy()), K, "exact")


@pytest.fixture(scope="module")
def g4_exact(oracle_pool):
    """The 8192 x 7168 x 7168 exact-kind product's operands and the oracle's
    bf16 output bits for every row, computed once on spawned workers (one
    512-row block of A each; a block starts on a 128-row tile, so its tiled
    scales are a contiguous slice)."""
    wl = workloads.GEMM_CONFIGS["G4_M8192_N7168_K7168"]
    a, b, sfa, sfb = operands(wl.M, wl.N, wl.K, wl.seed, "exact")
    an, bn, san, sbn = a.numpy(), b.numpy(), sfa.numpy(), sfb.numpy()
    tile_bytes = (wl.K // 64) * 512                        # one 128-row tile of NVFP4 scales
    blk = 512
    tasks = [(an[r0:r0 + blk], bn, san[r0 // 128 * tile_bytes:(r0 + blk) // 128 * tile_bytes], sbn,
              blk, wl.N, wl.K, "nvfp4") for r0 in range(0, wl.M, blk)]
    bits = np.concatenate(oracle_pool.map(acceptance.gemm_block_bits_task, tasks, chunksize=1))
    return wl, (a, b, sfa, sfb), bits


@pytest.mark.parametrize("variant", [-1] + VARIANTS)
def test_gemm_full_size_every_row(variant, g4_exact):
    """The 8192 x 7168 x 7168 product in the launch configuration the
    benchmark times (automatic variant) and in each tile schedule:
    exact-kind operands, every output element bit-exact."""
    wl, ops, want = g4_exact
    got = gpu_gemm(*ops, variant=variant)
    got_bits = got.view(torch.int16).cpu().numpy().view(np.uint16)
    bad = np.argwhere(got_bits != want)
    assert bad.size == 0, f"{len(bad)} of {want.size} outputs differ, first at {bad[:4].tolist()}"


@pytest.mark.parametrize("K", [2048, 1568])
@pytest.mark.parametrize("variant", [-1, 0, 2, 3])
def test_gemm_consumes_the_fused_producer_with_pdl(K, variant):
    """The fused op writes A and its tiled scales, fp4_quantize writes B, and the
    GEMM is launched as a programmatic dependent of the quantize kernel.  The
    oracle runs the same chain on the CPU; the producer's bytes equal the
    oracle's (up to boundary cases, none expected here), so the product is
    checked against the oracle's bound.  K = 1568: 98 scale blocks per row
    (two k-padding scales in the last tile, written as zero by the producers)
    and a last K block of 32 codes."""
    M, N = 300, 512
    wl = workloads.Workload("chain", M, K, "bf16", "nvfp4", "swizzled", 1e-6, seed=31)
    x, r, w = workloads.make_inputs(wl, "cpu")
    wmat = workloads.make_rows(workloads.Workload("wmat", N, K, "bf16", "nvfp4", "swizzled",
                                                  1e-6, seed=32), "x", 0, N, "cpu")
    oa = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                      wl.eps, "bf16", "nvfp4", "swizzled")
    ob = oracle.quantize(wmat.float().numpy(), "nvfp4", "swizzled")
    g = oracle.gemm_bf16(oa.packed, ob.packed, oa.sf_swizzled, ob.sf_swizzled, M, N, K)

    xr, rr = x.cuda(), r.clone().cuda()
    pa, sa = fq.add_rmsnorm_fp4quant(xr, rr, w.cuda(), eps=wl.eps, fmt="nvfp4",
                                     sf_layout="swizzled")
    pb, sb = fq.quantize_fp4(wmat.cuda(), fmt="nvfp4", sf_layout="swizzled")
    got = fq.gemm_nvfp4_bf16(pa, pb, sa, sb, pdl=True, variant=variant)
    torch.cuda.synchronize()
    same_a = np.array_equal(pa.cpu().numpy(), oa.packed) and np.array_equal(
        sa.cpu().numpy(), oa.sf_swizzled)
    same_b = np.array_equal(pb.cpu().numpy(), ob.packed) and np.array_equal(
        sb.cpu().numpy(), ob.sf_swizzled)
    assert same_a and same_b, "producer bytes differ from the oracle's"
    check(got, g, K, "random")


@pytest.mark.parametrize("M,N,K,variant,fmt", [(41, 4608, 1536, -1, "nvfp4"),
                                               (41, 1536, 6144, -1, "nvfp4"),
                                               (300, 512, 1568, 0, "nvfp4"),
                                               (300, 512, 1568, 4, "nvfp4"),
                                               (256, 768, 2048, 3, "nvfp4"),
                                               (41, 4608, 1536, -1, "mxfp4"),
                                               (300, 512, 1600, 4, "mxfp4")])
def test_gemm_static_weights_pdl2(M, N, K, variant, fmt):
    """A decode step's chain with static weights: B is quantized once and
    synchronised; then, three times, the fused op updates the residual and
    writes A, and the GEMM is launched with pdl = 2 (its B copies start before
    the dependency wait).  Every step's product matches the oracle GEMM of the
    operands that step's producer wrote."""
    steps = 3
    wl = workloads.Workload("static_b", M, K, "bf16", fmt, "swizzled", 1e-6, seed=M + K)
    x, r, w = workloads.make_inputs(wl, "cpu")
    wmat = workloads.make_rows(workloads.Workload("wmat_s", N, K, "bf16", fmt, "swizzled",
                                                  1e-6, seed=N + 5), "x", 0, N, "cpu")
    ob = oracle.quantize(wmat.float().numpy(), fmt, "swizzled")
    pb, sb = fq.quantize_fp4(wmat.cuda(), fmt=fmt, sf_layout="swizzled")
    torch.cuda.synchronize()
    xr, rr, wr = x.cuda(), r.clone().cuda(), w.cuda()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())   # the inputs' uploads
    outs = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            pa, sa = fq.add_rmsnorm_fp4quant(xr, rr, wr, eps=wl.eps, fmt=fmt,
                                             sf_layout="swizzled", pdl=True, stream=stream)
            outs.append((pa, sa, fq.gemm_nvfp4_bf16(pa, pb, sa, sb, pdl=2, variant=variant,
                                                    stream=stream, fmt=fmt)))
    stream.synchronize()
    assert np.array_equal(pb.cpu().numpy(), ob.packed)
    assert np.array_equal(sb.cpu().numpy(), ob.sf_swizzled)
    # each step's product against the oracle GEMM of the bytes that step's
    # producer wrote (the producer's own parity is tested on its own)
    for pa, sa, got in outs:
        g = oracle.gemm_bf16(pa.cpu().numpy(), ob.packed, sa.cpu().numpy(), ob.sf_swizzled,
                             M, N, K, fmt=fmt)
        check(got, g, K, "random")


@pytest.mark.parametrize("variant", [-1, 2, 3])
def test_gemm_consumes_the_mxfp4_producer(variant):
    """The headline producer configuration (bf16 rows with outlier columns,
    MXFP4, tiled scales) feeding the MXFP4 GEMM with PDL, against the oracle's
    chain."""
    M, N, K = 256, 384, 7168
    wl = workloads.Workload("chain_mx", M, K, "bf16", "mxfp4", "swizzled", 1e-6,
                            outlier_frac=0.01, seed=33)
    x, r, w = workloads.make_inputs(wl, "cpu")
    wmat = workloads.make_rows(workloads.Workload("wmat_mx", N, K, "bf16", "mxfp4", "swizzled",
                                                  1e-6, seed=34), "x", 0, N, "cpu")
    oa = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                      wl.eps, "bf16", "mxfp4", "swizzled")
    ob = oracle.quantize(wmat.float().numpy(), "mxfp4", "swizzled")
    g = oracle.gemm_bf16(oa.packed, ob.packed, oa.sf_swizzled, ob.sf_swizzled, M, N, K,
                         fmt="mxfp4")
    pa, sa = fq.add_rmsnorm_fp4quant(x.cuda(), r.clone().cuda(), w.cuda(), eps=wl.eps,
                                     fmt="mxfp4", sf_layout="swizzled")
    pb, sb = fq.quantize_fp4(wmat.cuda(), fmt="mxfp4", sf_layout="swizzled")
    got = fq.gemm_nvfp4_bf16(pa, pb, sa, sb, pdl=True, fmt="mxfp4", variant=variant)
    torch.cuda.synchronize()
    assert np.array_equal(pa.cpu().numpy(), oa.packed)
    assert np.array_equal(sa.cpu().numpy(), oa.sf_swizzled)
    assert np.array_equal(pb.cpu().numpy(), ob.packed)
    assert np.array_equal(sb.cpu().numpy(), ob.sf_swizzled)
    check(got, g, K, "random")


# ---------------------------------------------------------------------------
# GELU epilogues
# ---------------------------------------------------------------------------
import parity  # noqa: E402


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (41, 4608, 1536), (300, 520, 768),
                                   (77, 264, 352)])
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_gemm_gelu_bf16(M, N, K, variant):
    """GELU(alpha * product + bias) in bf16.  Exact-kind operands make the
    GELU argument exact; the GPU's erff-based GELU and one bf16 rounding keep
    every output within one bf16 step of the exact value."""
    a, b, sfa, sfb = operands(M, N, K, seed=11 * M + N, kind="exact")
    bias = bf16_values(N, 13, 4, (N,))
    got = fq.gemm_nvfp4_gelu(a.cuda(), b.cuda(), sfa.cuda(), sfb.cuda(), alpha=0.125,
                             bias=bias.cuda(), variant=variant)
    torch.cuda.synchronize()
    g = oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.125, bias=bias.float().numpy(),
                    gelu_act=True)
    got64 = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got64 - g.exact)
    tol = 2.0 ** -8 * np.abs(g.exact) + 2.0 ** -20
    assert np.all(err <= tol), f"{(err > tol).sum()} outputs off, first {np.argwhere(err > tol)[:4]}"


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (300, 528, 768), (41, 4608, 1536),
                                   (77, 272, 352)])
@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_gemm_gelu_nvfp4_output(M, N, K, variant):
    """The FP4-output epilogue against the oracle's quantization of the same
    GELU values, with the producer's acceptance rule (codes and scale bytes
    exact except within 1e-5 of a rounding boundary; tiled padding zero).  N =
    528 leaves a partial last group of four scales (k padding), M = 300 and 41
    leave padding rows."""
    a, b, sfa, sfb = operands(M, N, K, seed=17 * M + N, kind="exact")
    bias = bf16_values(N, 19, 4, (N,))
    outs = fq.gemm_nvfp4_gelu(a.cuda(), b.cuda(), sfa.cuda(), sfb.cuda(), alpha=0.25,
                              bias=bias.cuda(), out_format="nvfp4", variant=variant)
    torch.cuda.synchronize()
    o = oracle.gemm_gelu_nvfp4(a.numpy(), b.numpy(), sfa.numpy(), sfb.numpy(), M, N, K,
                               alpha=0.25, bias=bias.float().numpy())
    g = parity.fetch(outs, None, "swizzled", None, M=M)
    parity.compare(g, o, "nvfp4", "swizzled", "bf16", M, N)


def test_gemm_gelu_nvfp4_feeds_the_next_gemm():
    """Two chained projections: the first emits NVFP4 + tiled scales, the
    second consumes them as its A operand (PDL), against the oracle's chain."""
    M, N1, N2, K = 192, 512, 256, 1024
    a, b1, sfa, sfb1 = operands(M, N1, K, seed=23, kind="exact")
    _, b2, _, sfb2 = operands(N2, N2, N1, seed=29, kind="random")
    b2 = b2[:N2]
    pk, sf = fq.gemm_nvfp4_gelu(a.cuda(), b1.cuda(), sfa.cuda(), sfb1.cuda(), alpha=0.25,
                                out_format="nvfp4")
    got = fq.gemm_nvfp4_bf16(pk, b2.cuda(), sf, sfb2.cuda(), pdl=True)
    torch.cuda.synchronize()
    o1 = oracle.gemm_gelu_nvfp4(a.numpy(), b1.numpy(), sfa.numpy(), sfb1.numpy(), M, N1, K,
                                alpha=0.25)
    assert np.array_equal(pk.cpu().numpy(), o1.packed), "first projection's codes differ"
    assert np.array_equal(sf.cpu().numpy(), o1.sf_swizzled), "first projection's scales differ"
    g2 = oracle.gemm_bf16(o1.packed, b2.numpy(), o1.sf_swizzled, sfb2.numpy(), M, N2, N1)
    check(got, g2, N1, "random")


def test_gemm_gelu_nvfp4_rejects_split_k():
    a, b, sfa, sfb = operands(128, 128, 256, 1, "exact")
    with pytest.raises(fq.Fp4Error):
        fq.gemm_nvfp4_gelu(a.cuda(), b.cuda(), sfa.cuda(), sfb.cuda(), out_format="nvfp4",
                           variant=4)


def test_gemm_alternating_ring_depths():
    """A launch needing a deep ring (41 x 4608 x 1536: one wave, six stages),
    then a shallow one, then the deep one again: the kernel's shared-memory
    limit must not have been lowered in between."""
    for (M, N, K) in [(41, 4608, 1536), (300, 520, 768), (41, 4608, 1536), (8, 16, 256)]:
        a, b, sfa, sfb = operands(M, N, K, seed=M + K, kind="exact")
        got = gpu_gemm(a, b, sfa, sfb, variant=0)
        check(got, oracle_gemm(a, b, sfa, sfb, M, N, K), K, "exact")
