"""GPU parity of the standalone quantize (fp4_quantize) against the oracle's
quantize(), every format, layout and dtype, ragged shapes, global scale."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    fq.lib()


@pytest.mark.parametrize("M,H", [(1, 32), (3, 80), (130, 208), (1000, 1536), (257, 5120),
                                 (41, 7168), (129, 8224), (64, 17408), (5, 65536)])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "e4m3b32"])
@pytest.mark.parametrize("layout", ["rowmajor", "swizzled", "both"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quantize_parity(M, H, fmt, layout, dtype):
    if H % oracle.block_size(fmt):
        pytest.skip("H not a multiple of the block")
    wl = workloads.Workload("q", M, H, dtype, fmt, layout, 0.0, x_std=3.0, seed=M + H)
    x = workloads.make_rows(wl, "x", 0, M)
    o = oracle.quantize(x.float().numpy(), fmt, layout)
    g = parity.run_quantize(x.cuda(), fmt, layout)
    parity.compare(g, o, fmt, layout, dtype, M, H)
    if layout != "both":
        parity.check_dequant(g, M, H, fmt, layout)


@pytest.mark.parametrize("fmt", ["nvfp4", "e4m3b32", "mxfp4"])
def test_quantize_global_scale(fmt):
    M, H = 300, 4096
    wl = workloads.Workload("qg", M, H, "bf16", fmt, "swizzled", 0.0, x_std=2.0, seed=7)
    x = workloads.make_rows(wl, "x", 0, M)
    gs = float(np.float32(448.0 * 6.0 / x.float().abs().max().item()))
    o = oracle.quantize(x.float().numpy(), fmt, "swizzled", gs)
    g = parity.run_quantize(x.cuda(), fmt, "swizzled", global_scale=gs)
    parity.compare(g, o, fmt, "swizzled", "bf16", M, H)


def test_quantize_three_d_and_empty():
    x = torch.randn(2, 3, 256, device="cuda").to(torch.bfloat16)
    p, s = fq.quantize_fp4(x, fmt="nvfp4", sf_layout="rowmajor")
    assert p.shape == (2, 3, 128) and s.shape == (2, 3, 16)
    p2, s2 = fq.quantize_fp4(x.view(6, 256), fmt="nvfp4", sf_layout="rowmajor")
    torch.cuda.synchronize()
    assert torch.equal(p.view(6, 128), p2) and torch.equal(s.view(6, 16), s2)
    e = torch.empty(0, 256, device="cuda", dtype=torch.float16)
    p, s = fq.quantize_fp4(e, fmt="mxfp4", sf_layout="swizzled")
    assert p.numel() == 0 and s.numel() == 0


def _sample_rows(M, seed, n=96):
    fixed = {0, 1, 31, 32, 127, 128, 129, M // 2, M - 129, M - 128, M - 2, M - 1}
    rng = np.random.default_rng(seed)
    rand = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    return np.array(sorted(r for r in fixed | rand if 0 <= r < M), dtype=np.int64)


@pytest.mark.parametrize("name", ["C3_M8192_H7168_bf16_mxfp4_swizzled_outliers",
                                  "C4_M16384_H5120_fp16_nvfp4_both",
                                  "C5_M32768_H1536_bf16_nvfp4_swizzled",
                                  "C5_M32768_H6144_bf16_nvfp4_swizzled",
                                  "C5_M32768_H17408_bf16_mxfp4_swizzled",
                                  "C5_M32768_H32768_bf16_nvfp4_swizzled"])
def test_quantize_full_size_sampled(name):
    """The benchmarked quantize shapes at full size, in the launch the
    benchmark times: sampled rows (tile edges, first/last, seeded random)
    against the oracle, every padding byte of the tiled buffer checked."""
    wl = workloads.CONFIGS[name]
    x = workloads.make_inputs(wl, "cuda")[0]
    rows = _sample_rows(wl.M, wl.seed)
    xs = x.index_select(0, torch.from_numpy(rows).cuda()).float().cpu().numpy()
    g = parity.run_quantize(x, wl.fmt, wl.sf_layout, rows=rows)
    o = oracle.quantize(xs, wl.fmt, wl.sf_layout)
    parity.compare(g, o, wl.fmt, wl.sf_layout, wl.dtype, wl.M, wl.H)
