"""Host-side multi-rank helpers (one process per GPU).

Attention over a batch of sequences has no exchange step: every (sequence,
KV head) unit is independent, so ranks split the batch and never talk on the
data path. The only collectives are the timing barrier and the max over
ranks of the elapsed time.
"""
from __future__ import annotations

import os
from typing import List, Sequence


def rank_world() -> tuple:
    """(rank, world size, local rank) from the torchrun environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def partition_by_cost(costs: Sequence[int], world: int) -> List[List[int]]:
    """Split sequence indices over ``world`` ranks, balancing the summed cost.

    Longest-processing-time order: sequences by decreasing cost, each to the
    rank with the least load so far (ties to the lower rank). Every index
    appears in exactly one part; parts are returned sorted.
    """
    if world <= 0:
        raise ValueError("world must be positive")
    load = [0] * world
    parts: List[List[int]] = [[] for _ in range(world)]
    order = sorted(range(len(costs)), key=lambda i: (-int(costs[i]), i))
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        parts[r].append(i)
        load[r] += int(costs[i])
    return [sorted(p) for p in parts]


def max_over_ranks(value: float, device=None) -> float:
    """All-reduce MAX of a float over the default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None) -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()
