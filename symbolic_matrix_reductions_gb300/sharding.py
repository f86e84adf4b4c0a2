"""Row sharding of one reduction problem over several GPUs (one process per GPU).

Every reduction here is independent along i (the rows of x): row i's output needs
x_i and the whole of y, b, and nothing from any other row.  So one problem splits
over R ranks by contiguous row slices, with no exchange on the data path: rank r
takes rows [M r / R, M (r + 1) / R) of x (and of the upstream gradient g), calls
the unchanged C ABI on its own GPU with all of y and b, and writes the matching
rows of the caller-owned output, as the tiling manager of the GitHub issue
"Transparent interface for billion-scale matrices" splits a tall product over
GPUs and fills the blocks of ``out=``.  A collective is used only to bring the
slices together where the caller wants the whole output on one rank.

Ranks whose slice is empty (M < R) call nothing and return an empty slice.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class RowShard:
    """Rows [start, stop) of an M-row problem owned by `rank` of `world`."""
    rank: int
    world: int
    M: int
    start: int
    stop: int

    @property
    def rows(self) -> int:
        return self.stop - self.start

    def take(self, a):
        """This rank's rows of a row-major array or tensor with M rows (a view)."""
        return a[self.start:self.stop]


def row_shard(M: int, world: int, rank: int) -> RowShard:
    """Contiguous, balanced slice of M rows for `rank` of `world` (sizes differ by at
    most one; the slices cover [0, M) in rank order without overlap)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} out of range for world size {world}")
    if M < 0:
        raise ValueError(f"M must be >= 0, got {M}")
    return RowShard(rank, world, M, (M * rank) // world, (M * (rank + 1)) // world)


def all_shards(M: int, world: int):
    return [row_shard(M, world, r) for r in range(world)]


def gather_rows(local, shard: RowShard, group=None):
    """Concatenates every rank's slice in rank order on every rank (torch.distributed
    all-gather of the ragged slices, padded to the largest).  `local` is a torch tensor
    whose first dimension is shard.rows; the result has shard.M rows."""
    import torch
    import torch.distributed as dist

    world = shard.world
    if world == 1:
        return local
    sizes = [s.rows for s in all_shards(shard.M, world)]
    cap = max(sizes)
    pad = torch.zeros((cap,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    pad[:shard.rows] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:n] for p, n in zip(parts, sizes)], dim=0)
