"""The debug build (libfp4q_debug.so, include/fp4q.h "Debug build") on the GPU:

  * bounds checks: every global address the fused, quantize and GEMM kernels
    compute is compared with the extent of its buffer; over the parity grid's
    shapes, every kernel path and every GEMM schedule, the violation counter
    stays 0 and the outputs equal the default build's byte for byte; with the
    extents shrunk by one byte the counter rises for every kind of launch, so
    the checks do see the accesses at the end of each buffer;
  * timeouts: a chosen CTA arrives on a stage's barrier for a copy it never
    issues (nothing is left in flight), every bounded wait is cut to a few
    microseconds, and the kernel's timeout path runs: the device status word
    reads FP4_ERR_TIMEOUT, the rows (fused) or tiles (GEMM) of that CTA are
    marked, every other row or tile equals the oracle, and the next call on
    the same context runs normally.
No kernel faults, traps or spins without a bound here."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import parity
from test_gemm_gpu import oracle_gemm, operands

pytestmark = pytest.mark.gpu

DEFAULT_WAIT = 2_000_000_000
SHORT_WAIT = 20_000          # about 10 us at 2 GHz


@pytest.fixture(scope="module")
def D():
    fbuild.build()
    fbuild.build(debug=True)
    fq.lib()
    L = fq.debug_lib()
    assert L.fp4_debug_build() == 1
    yield L
    L.fp4_debug_configure(DEFAULT_WAIT, 0, 0, -1, -1, None)


def configure(D, wait=DEFAULT_WAIT, shrink=0, drop_kernel=0, drop_cta=-1, drop_iter=-1,
              counter=None):
    st = D.fp4_debug_configure(wait, shrink, drop_kernel, drop_cta, drop_iter,
                               counter.data_ptr() if counter is not None else None)
    assert st == 0


def _fused(L, x, r, w, fmt, layout, status=None):
    with fq.using_library(L):
        outs = fq.add_rmsnorm_fp4quant(x, r, w, fmt=fmt, sf_layout=layout, status=status)
    torch.cuda.synchronize()
    return outs


# every fused kernel path: register-resident rows (also one row per warp, and
# long batches), cluster rows, the TMA ring
FUSED_SHAPES = [(1, 64), (3, 80), (127, 208), (129, 1536), (130, 5120), (129, 7168),
                (41, 17408), (1, 32768), (2, 65536), (5000, 64), (2049, 208), (1999, 1536),
                (700, 7168), (613, 17408), (333, 32768), (20000, 1536), (2500, 7168)]


def test_checks_find_nothing_and_change_nothing(D):
    """Debug build over the shapes: counter 0, outputs equal the default
    build's (both libraries run on copies of the same inputs)."""
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    configure(D, counter=counter)
    kinds = set()
    for M, H in FUSED_SHAPES:
        for fmt in ("nvfp4", "mxfp4", "e4m3b32"):
            if H % oracle.block_size(fmt):
                continue
            for layout in ("rowmajor", "swizzled", "both"):
                wl = workloads.Workload("d", M, H, "bf16", fmt, layout, 1e-6, seed=M + H)
                x, r, w = workloads.make_inputs(wl, "cuda")
                r1, r2 = r.clone(), r.clone()
                a = _fused(fq.lib(), x, r1, w, fmt, layout)
                b = _fused(D, x, r2, w, fmt, layout)
                assert torch.equal(r1, r2), (M, H, fmt, layout)
                for ta, tb in zip(a, b):
                    assert torch.equal(ta, tb), (M, H, fmt, layout)
                kinds.add(fq.fp4_launch_shape(M, H, 0, fq.FP4_NVFP4 if fmt == "nvfp4" else
                                              fq.FP4_MXFP4, 1)["kernel"])
        # the standalone quantize on the same rows
        x = workloads.make_rows(workloads.Workload("q", M, H, "bf16", "nvfp4", "both", 1e-6,
                                                   seed=H), "x", 0, M, "cuda")
        with fq.using_library(D):
            qd = fq.quantize_fp4(x, fmt="nvfp4", sf_layout="both")
        qr = fq.quantize_fp4(x, fmt="nvfp4", sf_layout="both")
        torch.cuda.synchronize()
        for ta, tb in zip(qd, qr):
            assert torch.equal(ta, tb), ("quantize", M, H)
    assert kinds >= {"fused_direct_kernel", "fused_tma_kernel"}, kinds
    # the GEMM: every schedule, both operand formats, the epilogues
    for (M, N, K) in [(128, 128, 256), (300, 520, 768), (41, 1536, 6144), (1024, 1024, 1024)]:
        for fmt in ("nvfp4", "mxfp4"):
            a, b, sfa, sfb = [t.cuda() for t in operands(M, N, K, seed=M + N, kind="random",
                                                         fmt=fmt)]
            for variant in range(5):
                ref = fq.gemm_nvfp4_bf16(a, b, sfa, sfb, variant=variant, fmt=fmt)
                with fq.using_library(D):
                    got = fq.gemm_nvfp4_bf16(a, b, sfa, sfb, variant=variant, fmt=fmt)
                torch.cuda.synchronize()
                assert torch.equal(ref.view(torch.int16), got.view(torch.int16)), \
                    (M, N, K, fmt, variant)
        if N % 16 == 0:
            a, b, sfa, sfb = [t.cuda() for t in operands(M, N, K, seed=N, kind="random")]
            ref = fq.gemm_nvfp4_gelu(a, b, sfa, sfb, out_format="nvfp4")
            with fq.using_library(D):
                got = fq.gemm_nvfp4_gelu(a, b, sfa, sfb, out_format="nvfp4")
            torch.cuda.synchronize()
            assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1]), (M, N, K)
    torch.cuda.synchronize()
    assert int(counter.item()) == 0


def _count(D, fn):
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    configure(D, wait=SHORT_WAIT, shrink=1, counter=counter)
    try:
        with fq.using_library(D):
            fn()
        torch.cuda.synchronize()
    finally:
        configure(D)
    return int(counter.item())


@pytest.mark.parametrize("M,H,fmt,layout", [
    (129, 1536, "nvfp4", "rowmajor"),     # register-resident rows
    (41, 17408, "nvfp4", "swizzled"),     # cluster rows
    (333, 32768, "mxfp4", "both"),        # TMA ring (bulk-copy sources checked)
    (20000, 1536, "nvfp4", "swizzled"),   # persistent stream kernel
])
def test_shrunk_extents_are_caught_fused(D, M, H, fmt, layout):
    wl = workloads.Workload("s", M, H, "bf16", fmt, layout, 1e-6, seed=1)
    x, r, w = workloads.make_inputs(wl, "cuda")
    assert _count(D, lambda: fq.add_rmsnorm_fp4quant(x, r, w, fmt=fmt, sf_layout=layout)) > 0
    xq = x.clone()
    assert _count(D, lambda: fq.quantize_fp4(xq, fmt=fmt, sf_layout=layout)) > 0


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_shrunk_extents_are_caught_gemm(D, variant):
    M, N, K = 256, 512, 2048
    a, b, sfa, sfb = [t.cuda() for t in operands(M, N, K, seed=3, kind="random")]
    assert _count(D, lambda: fq.gemm_nvfp4_bf16(a, b, sfa, sfb, variant=variant)) > 0
    if variant != 4:
        assert _count(D, lambda: fq.gemm_nvfp4_gelu(a, b, sfa, sfb, out_format="nvfp4",
                                                    variant=variant)) > 0


def test_fused_timeout_marks_the_ctas_rows(D):
    """TMA-ring kernel: CTA 0 never issues its copies of ring iteration 1."""
    M, H, fmt = 1024, 32768, "nvfp4"
    shape = fq.fp4_launch_shape(M, H, 0, fq.FP4_NVFP4, fq.FP4_SF_BOTH)
    assert shape["kernel"] == "fused_tma_kernel"
    G, R = shape["ctas"], shape["slices_per_cta"]
    groups = -(-M // R)
    assert groups > G, "CTA 0 must own more than one row group"
    failed = sorted(g * R + q for g in range(G, groups, G) for q in range(R) if g * R + q < M)
    wl = workloads.Workload("t", M, H, "bf16", fmt, "both", 1e-6, seed=9)
    x, r, w = workloads.make_inputs(wl, "cuda")
    r0 = r.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    configure(D, wait=SHORT_WAIT, drop_kernel=1, drop_cta=0, drop_iter=1)
    try:
        packed, sf, sf_rm = _fused(D, x, r, w, fmt, "both", status=status)
    finally:
        configure(D)
    with fq.using_library(D):
        assert fq.read_device_status(status) == fq.FP4_ERR_TIMEOUT
    nb = H // 16
    rm = sf_rm.cpu().numpy().reshape(M, nb)
    assert np.all(rm[failed] == 0xFF)
    tiled = sf.cpu().numpy()
    kk = np.arange(nb)[None, :]
    assert np.all(tiled[oracle.swizzled_sf_offset(np.array(failed)[:, None], kk, (nb + 3) // 4)]
                  == 0xFF)
    ok = np.setdiff1d(np.arange(M), failed)
    idx = torch.from_numpy(ok).cuda()
    o = oracle.add_rmsnorm_fp4_quant(x.index_select(0, idx).float().cpu().numpy(),
                                     r0.index_select(0, idx).float().cpu().numpy(),
                                     w.float().cpu().numpy(), 1e-6, "bf16", fmt, "both")
    g = parity.fetch((packed, sf, sf_rm), r, "both", ok)
    parity.compare(g, o, fmt, "both", "bf16", M, H, check_padding=False)
    # the context is still usable: the same call runs normally
    status.zero_()
    r2 = r0.clone()
    _fused(D, x, r2, w, fmt, "both", status=status)
    with fq.using_library(D):
        assert fq.read_device_status(status) == fq.FP4_OK


@pytest.mark.parametrize("variant,M,N,K,bad_tiles", [
    (0, 256, 384, 1024, [(0, 0)]),                 # one CTA per tile: tile (0, 0)
    (2, 512, 512, 1024, [(0, 0)]),                 # persistent: CTA 0 owns one tile
    (4, 41, 1536, 6144, [(0, 0)]),                 # split K: rank 0 of tile 0's cluster
])
def test_gemm_timeout_marks_the_ctas_tiles(D, variant, M, N, K, bad_tiles):
    a, b, sfa, sfb = operands(M, N, K, seed=M + K, kind="exact")
    dev = [t.cuda() for t in (a, b, sfa, sfb)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    configure(D, wait=SHORT_WAIT, drop_kernel=2, drop_cta=0, drop_iter=1)
    try:
        with fq.using_library(D):
            out = fq.gemm_nvfp4_bf16(*dev, variant=variant, status=status)
        torch.cuda.synchronize()
    finally:
        configure(D)
    with fq.using_library(D):
        assert fq.read_device_status(status) == fq.FP4_ERR_TIMEOUT
    got = out.float().cpu().numpy()
    want = oracle_gemm(a, b, sfa, sfb, M, N, K).out
    mask = np.zeros((M, N), bool)
    for mt, nt in bad_tiles:
        mask[mt * 128:(mt + 1) * 128, nt * 128:(nt + 1) * 128] = True
    assert np.all(np.isnan(got[mask]))
    assert np.array_equal(got[~mask], want[~mask])
    # next call on the same context: normal
    status.zero_()
    with fq.using_library(D):
        out2 = fq.gemm_nvfp4_bf16(*dev, variant=variant, status=status)
        assert fq.read_device_status(status) == fq.FP4_OK
    assert np.array_equal(out2.float().cpu().numpy(), want)


def test_gemm_fp4_output_timeout_marks_scales(D):
    M, N, K = 256, 256, 1024
    a, b, sfa, sfb = operands(M, N, K, seed=17, kind="exact")
    dev = [t.cuda() for t in (a, b, sfa, sfb)]
    packed = torch.empty(M, N // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(fq.fp4_sf_size_bytes(M, N, fq.FP4_NVFP4, fq.FP4_SF_SWIZZLED),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    configure(D, wait=SHORT_WAIT, drop_kernel=2, drop_cta=0, drop_iter=1)
    try:
        with fq.using_library(D):
            st = fq.fp4_gemm_ex(*[t.data_ptr() for t in dev], fq.FP4_NVFP4,
                                fq.FP4_EPI_GELU_NVFP4, 1.0, 0, 0, M, N, K, 0, packed.data_ptr(),
                                sf.data_ptr(), 0, 0, status.data_ptr(), 0)
        assert st == 0
        torch.cuda.synchronize()
    finally:
        configure(D)
    with fq.using_library(D):
        assert fq.read_device_status(status) == fq.FP4_ERR_TIMEOUT
    ref_packed, ref_sf = fq.gemm_nvfp4_gelu(*dev, out_format="nvfp4", variant=0)
    torch.cuda.synchronize()
    nb = N // 16
    offs = oracle.swizzled_sf_offset(np.arange(128)[:, None], np.arange(8)[None, :],
                                     (nb + 3) // 4)          # tile (0, 0): blocks 0..7
    s = sf.cpu().numpy()
    assert np.all(s[offs] == 0xFF)
    mask = np.zeros(s.size, bool)
    mask[offs.reshape(-1)] = True
    assert np.array_equal(s[~mask], ref_sf.cpu().numpy()[~mask])
    pk, rpk = packed.cpu().numpy(), ref_packed.cpu().numpy()
    assert np.all(pk[:128, :64] == 0)
    assert np.array_equal(pk[128:], rpk[128:]) and np.array_equal(pk[:128, 64:], rpk[:128, 64:])
