"""Multi-GPU host logic: one process per GPU, sequences partitioned by rank.

The decode path has no exchange step: a sequence's blocks, table and cache
live on one GPU.  Under torchrun each rank serves its own replica of the
workload (different seed, same shape) -- weak scaling with no collective on
the data path.  The only collectives are the timing barrier and the max of the
per-rank elapsed times.
"""
import dataclasses
import os

import torch
import torch.distributed as dist


def env():
    """(world_size, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica(workload, rank: int):
    """The rank's own copy of a workload: same shape, independent draws."""
    return dataclasses.replace(workload, replica=int(rank))


def shard_bounds(n_units: int, world: int, rank: int):
    """Contiguous [start, end) of n_units for this rank (sizes differ by <= 1)."""
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
