"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
element by element (acceptance rule in tests/parity.py).  Shapes span several
128-row scale tiles with ragged tails, every dtype / format / scale layout,
the cluster (split-row) path, and special rows."""
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
    torch.cuda.init()


def _wl(M, H, dtype, fmt, layout, eps=1e-6, seed=0, **kw):
    return workloads.Workload(f"t_{M}_{H}", M, H, dtype, fmt, layout, eps, seed=seed, **kw)


def _run_full(wl, x=None, r=None, w=None, global_scale=None):
    """Inputs on the CPU (or given), oracle on every row, GPU through the C ABI."""
    if x is None:
        x, r, w = workloads.make_inputs(wl, "cpu")
    o = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                     wl.eps, wl.dtype, wl.fmt, wl.sf_layout,
                                     1.0 if global_scale is None else global_scale)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    g = parity.run_gpu(xd, rd, wd, wl.eps, wl.fmt, wl.sf_layout, global_scale=global_scale)
    stats = parity.compare(g, o, wl.fmt, wl.sf_layout, wl.dtype, wl.M, wl.H)
    return g, o, stats


# short batches (cluster kernel for wide rows), then batches long enough that
# persistent CTAs loop over several row groups of the TMA ring (ragged last
# group, tiled padding rows)
SHAPES = [(1, 64), (3, 80), (127, 208), (300, 256), (129, 1536), (300, 4096), (130, 5120),
          (129, 7168), (41, 17408), (1, 32768), (2, 65536), (5, 6144),
          (5000, 64), (2049, 208), (1999, 1536), (700, 7168), (613, 17408), (333, 32768)]


@pytest.mark.parametrize("M,H", SHAPES)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "e4m3b32"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("layout", ["rowmajor", "swizzled", "both"])
def test_parity_grid(M, H, fmt, dtype, layout):
    if H % oracle.block_size(fmt):
        pytest.skip("H not a multiple of the block")
    wl = _wl(M, H, dtype, fmt, layout, seed=M * 7 + H)
    g, o, _ = _run_full(wl)
    if layout != "both":
        parity.check_dequant(g, M, H, fmt, layout)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_special_rows(fmt):
    """Zero rows, a one-hot row, constant rows, an eps-dominated row, negative
    and signed-zero values, huge and tiny magnitudes in one batch."""
    H = 256
    M = 10
    x = torch.zeros(M, H)
    r = torch.zeros(M, H)
    r[1, 0] = 1.0                                  # one-hot
    r[2] = 1.0                                     # constant
    r[3] = 2.0 ** -10                              # eps-dominated
    x[4] = -0.5
    r[4] = -1.5                                    # negative constant
    x[5, ::2] = -0.0
    r[5, ::2] = -0.0                               # -0 + -0 = -0 in the residual
    r[5, 1::2] = 3.0
    r[6] = torch.linspace(-1000, 1000, H)          # large magnitudes
    r[7] = torch.linspace(-1e-20, 1e-20, H)        # tiny magnitudes
    r[8, :16] = 1e4                                # one huge block among small ones
    r[8, 16:] = 1e-3
    x[9] = 1.0
    r[9] = 2.0 ** -8                               # bf16 tie in the residual add
    w = torch.ones(H)
    w[::3] = -1.25                                 # negative weights give -0 in y
    wl = _wl(M, H, "bf16", fmt, "both")
    bf = torch.bfloat16
    x, r, w = x.to(bf), r.to(bf), w.to(bf)
    # bf16 subnormals (below 2^-126) in the residual add of row 7
    sub = torch.arange(1, 65, dtype=torch.int16).view(torch.bfloat16)
    x[7, :64] = sub
    r[7, :64] = -sub.flip(0)
    g, o, _ = _run_full(wl, x, r, w)
    # the zero row: zero magnitudes everywhere; NVFP4 zero scales give 0x0
    # codes, MXFP4 (scale 2^-127) keeps the sign of -0 products (0x8)
    assert np.all((g.packed[0] & 0x77) == 0)
    if fmt == "nvfp4":
        assert np.all(g.packed[0] == 0)
    parity.check_dequant(parity.GpuOut(g.rows, g.residual_bits, g.packed, g.sf, None),
                         M, H, fmt, "swizzled")


def test_determinism_and_stream():
    """Two runs on the same inputs give identical bytes, on a side stream."""
    wl = _wl(300, 7168, "bf16", "mxfp4", "swizzled", seed=5)
    x, r, w = workloads.make_inputs(wl, "cuda")
    r0 = r.clone()
    s = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        rr = r0.clone()
        torch.cuda.current_stream().synchronize()
        with torch.cuda.stream(s):
            p, sf = fq.add_rmsnorm_fp4quant(x, rr, w, eps=1e-6, fmt="mxfp4", sf_layout="swizzled",
                                            stream=s)
        s.synchronize()
        outs.append((rr.cpu(), p.cpu(), sf.cpu()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


def test_outputs_stay_inside_their_buffers():
    """Canary bytes around every output buffer survive the call."""
    M, H = 129, 5120
    wl = _wl(M, H, "fp16", "nvfp4", "both", seed=9)
    x, r, w = workloads.make_inputs(wl, "cuda")
    pad = 4096
    canary = 0xA5
    n_pk = M * H // 2
    n_sw = fq.fp4_sf_size_bytes(M, H, fq.FP4_NVFP4, fq.FP4_SF_SWIZZLED)
    n_rm = M * (H // 16)
    pk = torch.full((n_pk + 2 * pad,), canary, dtype=torch.uint8, device="cuda")
    sw = torch.full((n_sw + 2 * pad,), canary, dtype=torch.uint8, device="cuda")
    rm = torch.full((n_rm + 2 * pad,), canary, dtype=torch.uint8, device="cuda")
    rbuf = torch.full((M * H + 2 * pad,), 7.0, dtype=torch.float16, device="cuda")
    rbuf[pad:pad + M * H] = r.reshape(-1)
    rv = rbuf[pad:pad + M * H].view(M, H)
    fq.add_rmsnorm_fp4quant(x, rv, w, eps=1e-5, fmt="nvfp4", sf_layout="both",
                            out_packed=pk[pad:pad + n_pk].view(M, H // 2),
                            out_sf=sw[pad:pad + n_sw], out_sf_rowmajor=rm[pad:pad + n_rm])
    torch.cuda.synchronize()
    for buf, n in ((pk, n_pk), (sw, n_sw), (rm, n_rm)):
        assert torch.all(buf[:pad] == canary) and torch.all(buf[pad + n:] == canary)
    assert torch.all(rbuf[:pad] == 7.0) and torch.all(rbuf[pad + M * H:] == 7.0)


def test_empty_batch_is_a_no_op():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    r = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    p, sf = fq.add_rmsnorm_fp4quant(x, r, w, fmt="nvfp4", sf_layout="swizzled")
    assert p.shape == (0, 128) and sf.numel() == 0


def test_three_d_input_matches_two_d():
    wl = _wl(6 * 7, 1536, "bf16", "nvfp4", "rowmajor", seed=11)
    x, r, w = workloads.make_inputs(wl, "cuda")
    r2 = r.clone()
    p2, s2 = fq.add_rmsnorm_fp4quant(x, r2, w)
    r3 = r.clone().view(6, 7, 1536)
    p3, s3 = fq.add_rmsnorm_fp4quant(x.view(6, 7, 1536), r3, w)
    torch.cuda.synchronize()
    assert p3.shape == (6, 7, 768) and s3.shape == (6, 7, 96)
    assert torch.equal(p2.view(6, 7, 768), p3) and torch.equal(r2.view(6, 7, 1536), r3)
    assert torch.equal(s2.view(6, 7, 96), s3)


def test_launch_shapes_cover_every_kernel():
    """The shapes above reach the TMA-ring kernel, the register-resident kernel
    and its cluster mode (so the parity grid exercises all three)."""
    s = fq.fp4_launch_shape(333, 32768, fq.FP4_DT_BF16, fq.FP4_NVFP4, fq.FP4_SF_SWIZZLED)
    assert s["kernel"] == "fused_tma_kernel" and s["stages"] >= 1
    s = fq.fp4_launch_shape(700, 7168, fq.FP4_DT_BF16, fq.FP4_MXFP4, fq.FP4_SF_SWIZZLED)
    assert s["kernel"] == "fused_direct_kernel" and s["cluster"] == 1
    s = fq.fp4_launch_shape(41, 17408, fq.FP4_DT_BF16, fq.FP4_NVFP4, fq.FP4_SF_SWIZZLED)
    assert s["kernel"] == "fused_direct_kernel" and s["cluster"] > 1
    s = fq.fp4_launch_shape(2, 65536, fq.FP4_DT_FP16, fq.FP4_MXFP4, fq.FP4_SF_ROWMAJOR)
    assert s["cluster"] >= 2


@pytest.mark.parametrize("M,H", [(129, 1536), (700, 7168), (41, 17408), (333, 32768)])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "e4m3b32"])
@pytest.mark.parametrize("gs", [2688.0 / 3.9, 0.37])
def test_global_scale(M, H, fmt, gs):
    """Device-resident global scale through every kernel (direct, cluster,
    TMA ring); UE8M0 scales ignore it."""
    wl = _wl(M, H, "bf16", fmt, "both", seed=3 * M + H)
    _run_full(wl, global_scale=gs)


@pytest.mark.parametrize("M,H", [(129, 1536), (700, 7168), (41, 17408), (333, 32768)])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_strided_rows_and_y_output(M, H, fmt, dtype):
    """Input and residual as column slices of wider matrices (row strides
    H + 64 and H + 128), y returned in the storage dtype: codes, scales and
    residual equal the oracle's, and y is the oracle's fp32 y rounded once
    (up to the midpoint rule of `parity.compare_y`);
    every kernel path (direct, cluster, TMA ring)."""
    wl = _wl(M, H, dtype, fmt, "both", seed=5 * M + H)
    x, r, w = workloads.make_inputs(wl, "cpu")
    o = oracle.add_rmsnorm_fp4_quant(x.float().numpy(), r.float().numpy(), w.float().numpy(),
                                     wl.eps, dtype, fmt, "both")
    xw = torch.full((M, H + 64), 3.0, dtype=x.dtype, device="cuda")
    rw = torch.full((M, H + 128), 5.0, dtype=x.dtype, device="cuda")
    xw[:, :H] = x.cuda()
    rw[:, 64:64 + H] = r.cuda()
    xv, rv = xw[:, :H], rw[:, 64:64 + H]
    packed, sf, sf_rm, y = fq.add_rmsnorm_fp4quant(xv, rv, w.cuda(), eps=wl.eps, fmt=fmt,
                                                   sf_layout="both", return_y=True)
    torch.cuda.synchronize()
    g = parity.fetch((packed, sf, sf_rm), rv, "both")
    parity.compare(g, o, fmt, "both", dtype, M, H)
    parity.compare_y(y.view(torch.int16).cpu().numpy().view(np.uint16), o.y, dtype)
    # the padding columns around the views are untouched
    assert torch.all(xw[:, H:] == 3.0) and torch.all(rw[:, :64] == 5.0)
    assert torch.all(rw[:, 64 + H:] == 5.0)
