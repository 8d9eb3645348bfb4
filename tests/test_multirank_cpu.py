"""The N > 1 path on the CPU: two gloo ranks each take their 128-row-aligned
shard of one batch, compute it (with the oracle: no GPU here), and rank 0
checks that the gathered shards equal the single-process result, including
the tiled scale buffer assembled from the ranks' byte ranges; and the bench's
max-over-ranks timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads
from rmsnorm_fp4_quant_gb300.sharding import shard_rows


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, M, H, fmt, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = workloads.Workload("shard", M, H, "bf16", fmt, "both", 1e-6, seed=21)
        sh = shard_rows(M, H, wl.block, world, rank)
        x = workloads.make_rows(wl, "x", sh.row0, sh.row1).float().numpy()
        r = workloads.make_rows(wl, "r", sh.row0, sh.row1).float().numpy()
        w = workloads.make_weight(wl).float().numpy()
        o = oracle.add_rmsnorm_fp4_quant(x, r, w, wl.eps, "bf16", fmt, "both")
        # local tiled buffer == the rank's byte range of the global one
        assert o.sf_swizzled.size == sh.sf_tiled1 - sh.sf_tiled0
        parts = [None] * world
        dist.all_gather_object(parts, (sh, o.packed, o.sf_rowmajor, o.sf_swizzled, o.residual))
        t = torch.tensor([1.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            xf = workloads.make_rows(wl, "x", 0, M).float().numpy()
            rf = workloads.make_rows(wl, "r", 0, M).float().numpy()
            full = oracle.add_rmsnorm_fp4_quant(xf, rf, w, wl.eps, "bf16", fmt, "both")
            packed = np.concatenate([p[1] for p in parts])
            sf_rm = np.concatenate([p[2] for p in parts])
            res = np.concatenate([p[4] for p in parts])
            tiled = np.zeros_like(full.sf_swizzled)
            for shp, _, _, sft, _ in parts:
                tiled[shp.sf_tiled0:shp.sf_tiled1] = sft
            ok = (np.array_equal(packed, full.packed) and np.array_equal(sf_rm, full.sf_rowmajor)
                  and np.array_equal(tiled, full.sf_swizzled) and np.array_equal(res, full.residual)
                  and float(t.item()) == float(world))
            with open(result_path, "w") as f:
                f.write("ok" if ok else "mismatch")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("M,H,fmt", [(300, 256, "nvfp4"), (129, 1536, "mxfp4")])
def test_two_rank_shards_match_single_process(tmp_path, M, H, fmt):
    path = str(tmp_path / "result.txt")
    mp.start_processes(_worker, args=(2, _free_port(), M, H, fmt, path), nprocs=2,
                       join=True, start_method="spawn")
    assert open(path).read() == "ok"


def test_shard_rows_cover_the_batch_on_tile_boundaries():
    for M in (1, 127, 128, 300, 8192, 16385):
        for world in (1, 2, 3, 8):
            shards = [shard_rows(M, 1536, 16, world, r) for r in range(world)]
            assert shards[0].row0 == 0 and shards[-1].row1 == M
            for a, b in zip(shards, shards[1:]):
                assert a.row1 == b.row0 and a.sf_tiled1 == b.sf_tiled0
            for s in shards:
                assert s.row0 % 128 == 0 or s.row0 == s.row1 == M   # empty tail shards
