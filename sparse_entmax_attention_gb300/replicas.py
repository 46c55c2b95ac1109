"""Multi-GPU runs of the decode step are independent replicas (the step has
no exchange between devices): one process per GPU, a barrier around the timed
region, and the slowest rank's step time as the job's step time."""

from __future__ import annotations

import torch
import torch.distributed as dist


def world() -> tuple[int, int]:
    if dist.is_available() and dist.is_initialized():
        return dist.get_rank(), dist.get_world_size()
    return 0, 1


def barrier() -> None:
    if world()[1] > 1:
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the value itself on one rank)."""
    if world()[1] == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
