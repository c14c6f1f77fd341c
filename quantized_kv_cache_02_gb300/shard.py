"""Data parallelism over sequences: one process per GPU, each holding a
contiguous shard of the global batch in its own caches.

Appends, flushes and the decode attention of one sequence read no other
sequence's state: each request of a batch owns its KV ("KV Cache 与自回归视频生成"
section 6.1), so a shard needs nothing from another rank and there is no
collective on the data path.  Ranks meet only
to time a step (a barrier on both sides) and to fold per-rank figures into
whole-job ones: the slowest rank's time and the sum of the units processed.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shard:
    """Global sequences ``[begin, begin + count)`` owned by ``rank``."""
    rank: int
    world: int
    begin: int
    count: int

    @property
    def seqs(self) -> range:
        return range(self.begin, self.begin + self.count)


def shard_range(global_batch: int, world: int, rank: int) -> Shard:
    """Contiguous, balanced split: the first ``global_batch % world`` ranks
    take one sequence more.  Raises ValueError on a bad rank or world size, or
    when a rank would get no sequence."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} out of range for world size {world}")
    if global_batch < world:
        raise ValueError(f"global batch {global_batch} leaves a rank of {world} without sequences")
    base, extra = divmod(global_batch, world)
    begin = rank * base + min(rank, extra)
    return Shard(rank, world, begin, base + (1 if rank < extra else 0))


def job_totals(local_units: float, local_ms: float, dist=None, device="cpu") -> tuple[float, float]:
    """Whole-job (units summed over ranks, time as the max over ranks).

    ``dist`` is an initialised ``torch.distributed`` (any backend whose
    all_reduce takes tensors on ``device``) or None for one process."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(local_units), float(local_ms)
    import torch
    units = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    ms = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(units, op=dist.ReduceOp.SUM)
    dist.all_reduce(ms, op=dist.ReduceOp.MAX)
    return units.item(), ms.item()
