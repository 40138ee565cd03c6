"""Data-parallel sharding of the attention forward pass across ranks.

Every (batch entry, head) pair is an independent problem: the h heads run in
parallel and are only concatenated afterwards (section 3.2.2 of "Attention Is
All You Need"), and batch entries never interact.  N ranks (one process per
GPU) therefore split the global batch into contiguous slices with no
collective on the data path; each rank runs the fused kernel on its own
slice, already resident in its own HBM.  The only collectives here are for
the host: the maximum of the per-rank step times (the job is as slow as its
slowest rank) and, for a caller that wants the whole output on every rank,
an all-gather of O and LSE.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_range(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """Batch entries [start, stop) owned by `rank`; the slices partition
    [0, global_batch) and differ in size by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of {world}")
    if global_batch < 0:
        raise ValueError("negative batch")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seeds(rank: int, base=(0, 1, 2, 3)) -> tuple[int, ...]:
    """Input-generator seeds for a rank's slice (rank 0 keeps the base seeds)."""
    return tuple(s + 1000 * rank for s in base)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over all ranks (identity without a process group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_batch(local: torch.Tensor, global_batch: int) -> torch.Tensor:
    """All-gather per-rank slices along dim 0 into the [global_batch, ...]
    tensor on every rank (slices may differ in size by one)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local
    world = dist.get_world_size()
    sizes = [shard_range(global_batch, world, r) for r in range(world)]
    longest = max(b - a for a, b in sizes)
    pad = torch.zeros((longest,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    pad[: local.shape[0]] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    return torch.cat([p[: b - a] for p, (a, b) in zip(parts, sizes)], dim=0)
