"""GPU parity on the five workload families at their full sizes, in the same
launch configuration the benchmark times (the C ABI picks it from M, H and
the format).  Every row is compared with the oracle: the batch is cut into
blocks of about 4M elements, each block's pristine inputs and the GPU's bytes
for it go to a pool of spawned processes that run the oracle and the
acceptance rule (tests/acceptance.py) on it, and the excused exceptions are
summed over the whole workload before the 1e-4 bound is applied.  The tiled
padding is checked over the whole buffer, the two scale layouts against each
other on every row, and small workloads also through the library's dequant."""
import numpy as np
import pytest
import torch

import acceptance
import oracle
import rmsnorm_fp4_quant_gb300 as fq
import workloads
from rmsnorm_fp4_quant_gb300 import build as fbuild

import parity

pytestmark = pytest.mark.gpu

BLOCK_ELEMS = 1 << 22
SMALL_ELEMS = 1 << 22       # at most this many elements: also checked through fp4_dequant


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    fq.lib()


def _bits16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_workload(wl: workloads.Workload, pool):
    small = wl.M * wl.H <= SMALL_ELEMS
    if small:
        xc, rc, wc = workloads.make_inputs(wl, "cpu")
        x, r, w = xc.cuda(), rc.cuda(), wc.cuda()
    else:
        x, r, w = workloads.make_inputs(wl, "cuda")
    r0 = r.clone()
    outs = fq.add_rmsnorm_fp4quant(x, r, w, eps=wl.eps, fmt=wl.fmt, sf_layout=wl.sf_layout)
    torch.cuda.synchronize()
    M, H = wl.M, wl.H
    nb = H // wl.block
    packed = outs[0].reshape(M, H // 2)
    sf = outs[1].cpu().numpy().reshape(-1)
    sf_rm = outs[2].cpu().numpy().reshape(M, nb) if wl.sf_layout == "both" else None
    if wl.sf_layout == "rowmajor":
        sf_rows = sf.reshape(M, nb)
    else:
        assert acceptance.tiled_padding_is_zero(sf, M, nb), "tiled padding bytes are not zero"
    ws = w.float().cpu().numpy()
    step = max(1, BLOCK_ELEMS // H)

    def task(a):
        b = min(M, a + step)
        if wl.sf_layout == "rowmajor":
            sc = sf_rows[a:b]
        else:
            mm = np.arange(a, b)[:, None]
            kk = np.arange(nb)[None, :]
            sc = sf[oracle.swizzled_sf_offset(mm, kk, (nb + 3) // 4)]
            if sf_rm is not None:
                assert np.array_equal(sf_rm[a:b], sc), f"scale layouts disagree in rows {a}.."
        return (_bits16(x[a:b]), _bits16(r0[a:b]), ws, wl.eps, wl.dtype, wl.fmt,
                _bits16(r[a:b]), packed[a:b].cpu().numpy(), sc)

    # blocks go to the workers a batch at a time, so host memory holds only
    # a couple of blocks per worker
    starts = list(range(0, M, step))
    batch = 32
    n_exc = n_el = 0
    for i in range(0, len(starts), batch):
        for e, n in pool.map(acceptance.fused_block_task, [task(a) for a in starts[i:i + batch]],
                             chunksize=1):
            n_exc += e
            n_el += n
    assert n_el == M * H
    assert n_exc <= acceptance.MAX_EXCEPTION_FRAC * n_el, f"{n_exc} exceptions in {n_el}"
    if small and wl.sf_layout != "both":
        g = parity.fetch(outs, r, wl.sf_layout)
        parity.check_dequant(g, M, H, wl.fmt, wl.sf_layout)
    return {"exceptions": n_exc, "elements": n_el}


@pytest.mark.parametrize("wl", [workloads.C1, workloads.C2, workloads.C3, workloads.C4],
                         ids=lambda w: w.name)
def test_named_configs(wl, oracle_pool, parity_log):
    stats = run_workload(wl, oracle_pool)
    parity_log.append((wl.name, stats["exceptions"], stats["elements"]))


@pytest.mark.parametrize("wl", workloads.sweep(), ids=lambda w: w.name)
def test_sweep(wl, oracle_pool, parity_log):
    stats = run_workload(wl, oracle_pool)
    parity_log.append((wl.name, stats["exceptions"], stats["elements"]))
