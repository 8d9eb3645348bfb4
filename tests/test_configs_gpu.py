"""GPU parity on the five workload families at their full sizes, in the same
launch configuration the benchmark times (the C ABI picks it from M, H and
the format).  Small cases are compared with the oracle on every row; large
ones on sampled rows (first/last rows, 128-row tile edges and seeded random
rows), plus properties checked on every row: the residual equals the
dtype-rounded sum of the pristine inputs, the two scale layouts agree, and
every padding byte of the tiled buffer is zero."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import parity

pytestmark = pytest.mark.gpu

FULL_ORACLE_ELEMS = 1 << 22


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    fq.lib()


def _sample_rows(M, n=96, seed=0):
    fixed = {0, 1, 31, 32, 127, 128, 129, M // 2, M - 129, M - 128, M - 2, M - 1}
    rng = np.random.default_rng(seed)
    rand = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    return np.array(sorted(r for r in fixed | rand if 0 <= r < M), dtype=np.int64)


def _residual_property(x, r0, r_new, dtype):
    """Every row: residual == rn_dtype(float(x) + float(r0)) (torch's own
    rounding cast), checked in row blocks to bound memory."""
    step = max(1, (1 << 26) // x.shape[1])
    for i in range(0, x.shape[0], step):
        want = (x[i:i + step].float() + r0[i:i + step].float()).to(dtype)
        assert torch.equal(want.view(torch.int16), r_new[i:i + step].view(torch.int16)), i


def run_workload(wl: workloads.Workload):
    big = wl.M * wl.H > FULL_ORACLE_ELEMS
    dev = "cuda"
    if big:
        x, r, w = workloads.make_inputs(wl, dev)
        rows = _sample_rows(wl.M, seed=wl.seed)
    else:
        xc, rc, wc = workloads.make_inputs(wl, "cpu")
        x, r, w = xc.to(dev), rc.to(dev), wc.to(dev)
        rows = np.arange(wl.M)
    r0 = r.clone()
    idx = torch.from_numpy(rows).to(dev)
    xs = x.index_select(0, idx).float().cpu().numpy()
    rs = r0.index_select(0, idx).float().cpu().numpy()
    ws = w.float().cpu().numpy()
    g = parity.run_gpu(x, r, w, wl.eps, wl.fmt, wl.sf_layout, rows=rows)
    o = oracle.add_rmsnorm_fp4_quant(xs, rs, ws, wl.eps, wl.dtype, wl.fmt, wl.sf_layout)
    stats = parity.compare(g, o, wl.fmt, wl.sf_layout, wl.dtype, wl.M, wl.H)
    _residual_property(x, r0, r, wl.torch_dtype)
    if not big and wl.sf_layout != "both":
        parity.check_dequant(g, wl.M, wl.H, wl.fmt, wl.sf_layout)
    return stats


@pytest.mark.parametrize("wl", [workloads.C1, workloads.C2, workloads.C3, workloads.C4],
                         ids=lambda w: w.name)
def test_named_configs(wl):
    run_workload(wl)


@pytest.mark.parametrize("wl", workloads.sweep(), ids=lambda w: w.name)
def test_sweep(wl):
    run_workload(wl)
