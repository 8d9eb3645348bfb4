"""Row sharding of one batch over several GPUs (host logic only).

Rows are independent and the weight is replicated, so a batch splits over
ranks with no data exchange.  Cuts fall on multiples of 128 rows: each rank
then owns whole 128-row tiles of the tiled scale layout, and its tiled scale
bytes are one contiguous range of the global buffer (tile m/128 starts at
(m/128) * nkt * 512), as are its rows of the residual, the codes and the
row-major scales.
"""
from __future__ import annotations

from typing import NamedTuple


class Shard(NamedTuple):
    row0: int          # first row of the rank
    row1: int          # one past the last row
    sf_tiled0: int     # byte range of the rank's tiles in the global tiled buffer
    sf_tiled1: int


def shard_rows(M: int, H: int, block: int, world: int, rank: int) -> Shard:
    """Rows [row0, row1) and tiled-scale bytes [sf_tiled0, sf_tiled1) of `rank`."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    tiles = (M + 127) // 128
    per, extra = divmod(tiles, world)
    t0 = rank * per + min(rank, extra)
    t1 = t0 + per + (1 if rank < extra else 0)
    nkt = ((H // block) + 3) // 4
    return Shard(min(M, t0 * 128), min(M, t1 * 128), t0 * nkt * 512, t1 * nkt * 512)
