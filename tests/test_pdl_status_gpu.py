"""Programmatic dependent launch and the device status word on the default
build, through the C ABI:

  * fused calls chained with pdl = 1, each reading the residual the previous
    one wrote (the dependency PDL must honour), equal the oracle applied the
    same number of times, on every kernel path (one row per warp, the
    register-resident kernel, cluster rows, the TMA ring);
  * fp4_quantize with pdl = 1 right after the fused op quantizes the residual
    that call wrote;
  * a call given a status word leaves it 0 when nothing timed out, and
    fp4_read_device_status reads it back (fused kernel paths and every GEMM
    schedule through fp4_gemm_ex)."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import parity
from test_gemm_gpu import check, operands, oracle_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    fq.lib()


@pytest.mark.parametrize("M,H,fmt", [(300, 1536, "nvfp4"), (257, 7168, "mxfp4"),
                                     (41, 17408, "nvfp4"), (333, 32768, "e4m3b32")])
def test_chained_calls_with_pdl(M, H, fmt):
    steps = 4
    wl = workloads.Workload("p", M, H, "bf16", fmt, "swizzled", 1e-6, seed=M + H)
    x, r, w = workloads.make_inputs(wl, "cpu")
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())   # the inputs' uploads
    outs = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            outs.append(fq.add_rmsnorm_fp4quant(xd, rd, wd, eps=wl.eps, fmt=fmt,
                                                sf_layout="swizzled", pdl=True, stream=stream))
    stream.synchronize()
    # the oracle, step by step on the residual it produced
    rk = r.float().numpy()
    for k in range(steps):
        o = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), rk, w.float().numpy(), wl.eps,
                                         "bf16", fmt, "swizzled")
        # each step wrote its own code and scale buffers; the residual is
        # checked after the last step (the steps before overwrote it in turn)
        g = parity.fetch(outs[k], rd if k == steps - 1 else None, "swizzled", M=M)
        parity.compare(g, o, fmt, "swizzled", "bf16", M, H)
        rk = o.residual


def test_quantize_with_pdl_reads_the_fused_output():
    M, H = 512, 6144
    wl = workloads.Workload("q", M, H, "bf16", "nvfp4", "swizzled", 1e-6, seed=5)
    x, r, w = workloads.make_inputs(wl, "cpu")
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())   # the inputs' uploads
    with torch.cuda.stream(stream):
        fq.add_rmsnorm_fp4quant(xd, rd, wd, fmt="nvfp4", sf_layout="swizzled", stream=stream)
        pq, sq = fq.quantize_fp4(rd, fmt="nvfp4", sf_layout="swizzled", pdl=True, stream=stream)
    stream.synchronize()
    h = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                     1e-6, "bf16", "nvfp4", "swizzled").residual
    o = oracle.quantize(h, "nvfp4", "swizzled")
    assert np.array_equal(pq.cpu().numpy(), o.packed)
    assert np.array_equal(sq.cpu().numpy(), o.sf_swizzled)


@pytest.mark.parametrize("M,H", [(129, 1536), (700, 7168), (41, 17408), (333, 32768)])
def test_status_word_stays_zero(M, H):
    wl = workloads.Workload("s", M, H, "bf16", "mxfp4", "both", 1e-6, seed=H)
    x, r, w = workloads.make_inputs(wl, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fq.add_rmsnorm_fp4quant(x, r, w, fmt="mxfp4", sf_layout="both", status=status)
    assert fq.read_device_status(status) == fq.FP4_OK
    assert int(status.item()) == 0


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_gemm_ex_status_and_result(variant, fmt):
    M, N, K = 300, 520, 2048
    a, b, sfa, sfb = operands(M, N, K, seed=N + variant, kind="exact", fmt=fmt)
    dev = [t.cuda() for t in (a, b, sfa, sfb)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fq.gemm_nvfp4_bf16(*dev, alpha=0.5, variant=variant, fmt=fmt, status=status)
    assert fq.read_device_status(status) == fq.FP4_OK
    check(out, oracle_gemm(a, b, sfa, sfb, M, N, K, alpha=0.5, fmt=fmt), K, "exact")


def test_gemm_ex_mxfp4_gelu_bf16():
    """The GELU epilogue on MXFP4 operands (reachable through fp4_gemm_ex)."""
    M, N, K = 256, 384, 1024
    a, b, sfa, sfb = operands(M, N, K, seed=3, kind="exact", fmt="mxfp4")
    dev = [t.cuda() for t in (a, b, sfa, sfb)]
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = fq.fp4_gemm_ex(*[t.data_ptr() for t in dev], fq.FP4_MXFP4, fq.FP4_EPI_GELU_BF16, 1.0,
                        0, 0, M, N, K, out.data_ptr(), 0, 0, -1, 0, 0, 0)
    assert st == 0
    torch.cuda.synchronize()
    g = oracle_gemm(a, b, sfa, sfb, M, N, K, fmt="mxfp4", gelu_act=True)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - g.exact) <= 2.0 ** -8 * np.abs(g.exact) + 2.0 ** -20)
