"""GPU parity of the standalone quantize (fp4_quantize) against the oracle's
quantize(), every format, layout and dtype, ragged shapes, global scale."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import acceptance
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


@pytest.mark.parametrize("name", ["C3_M8192_H7168_bf16_mxfp4_swizzled_outliers",
                                  "C4_M16384_H5120_fp16_nvfp4_both",
                                  "C5_M32768_H1536_bf16_nvfp4_swizzled",
                                  "C5_M32768_H6144_bf16_nvfp4_swizzled",
                                  "C5_M32768_H17408_bf16_mxfp4_swizzled",
                                  "C5_M32768_H32768_bf16_nvfp4_swizzled"])
def test_quantize_full_size_every_row(name, oracle_pool, parity_log):
    """The benchmarked quantize shapes at full size, in the launch the
    benchmark times: every row against the oracle (blocks of about 4M
    elements on spawned workers, exceptions summed over the workload), the
    two scale layouts against each other, every padding byte of the tiled
    buffer."""
    wl = workloads.CONFIGS[name]
    M, H = wl.M, wl.H
    nb = H // wl.block
    x = workloads.make_inputs(wl, "cuda")[0]
    outs = fq.quantize_fp4(x, fmt=wl.fmt, sf_layout=wl.sf_layout)
    torch.cuda.synchronize()
    packed = outs[0]
    sf = outs[1].cpu().numpy().reshape(-1)
    if wl.sf_layout == "rowmajor":
        rows_sf = sf.reshape(M, nb)
    else:
        assert acceptance.tiled_padding_is_zero(sf, M, nb)
    sf_rm = outs[2].cpu().numpy().reshape(M, nb) if wl.sf_layout == "both" else None
    step = max(1, (1 << 22) // H)

    def task(a):
        b = min(M, a + step)
        if wl.sf_layout == "rowmajor":
            sc = rows_sf[a:b]
        else:
            sc = sf[oracle.swizzled_sf_offset(np.arange(a, b)[:, None], np.arange(nb)[None, :],
                                              (nb + 3) // 4)]
            if sf_rm is not None:
                assert np.array_equal(sf_rm[a:b], sc), f"scale layouts disagree in rows {a}.."
        return (x[a:b].view(torch.int16).cpu().numpy().view(np.uint16), wl.dtype, wl.fmt,
                packed[a:b].cpu().numpy(), sc)

    starts = list(range(0, M, step))
    n_exc = n_el = 0
    for i in range(0, len(starts), 32):
        tasks = [task(a) for a in starts[i:i + 32]]
        for e, n in oracle_pool.map(acceptance.quantize_block_task, tasks, chunksize=1):
            n_exc += e
            n_el += n
    assert n_el == M * H
    assert n_exc <= acceptance.MAX_EXCEPTION_FRAC * n_el
    parity_log.append((name + " (quantize)", n_exc, n_el))
