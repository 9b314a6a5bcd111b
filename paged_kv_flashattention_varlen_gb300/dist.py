"""Host-side multi-rank helpers (one process per GPU).

Attention over a batch of sequences has no exchange step: every (sequence,
KV head) unit is independent, so ranks split the batch by sequences
(``partition_by_cost``) or by KV heads (``head_shard``, ``shard_heads``) and
never talk on the data path. The only collectives are the timing barrier and
the max over ranks of the elapsed time (and a gather of output heads where a
consumer wants every head on one rank).
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


def head_shard(n_heads_q: int, n_heads_kv: int, world: int, rank: int) -> tuple:
    """Head (tensor) sharding: rank ``rank`` of ``world`` owns a contiguous block
    of whole KV heads, [k0, k1), and the query heads that read them, [q0, q1) =
    [k0 G, k1 G) with G = n_heads_q / n_heads_kv (query head h reads KV head
    h / G). KV heads are dealt as evenly as possible (the first
    n_heads_kv % world ranks hold one more). Returns (q0, q1, k0, k1)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if n_heads_kv <= 0 or n_heads_q % n_heads_kv:
        raise ValueError("n_heads_q must be a multiple of n_heads_kv")
    g = n_heads_q // n_heads_kv
    base, extra = divmod(n_heads_kv, world)
    k0 = rank * base + min(rank, extra)
    k1 = k0 + base + (1 if rank < extra else 0)
    return k0 * g, k1 * g, k0, k1


def shard_heads(q, kv_pool, n_heads_q: int, n_heads_kv: int, world: int, rank: int, paged: bool = True):
    """This rank's slices of the query rows [total_q, Hq, D] and of the cache
    ([pages, 2, 64, Hkv, D] paged, or [2, rows, Hkv, D] contiguous), as
    contiguous tensors for the library (which takes dense layouts); the block
    table, lengths and query offsets are shared unchanged. Returns
    (q_rank, kv_rank, n_heads_q_rank, n_heads_kv_rank)."""
    q0, q1, k0, k1 = head_shard(n_heads_q, n_heads_kv, world, rank)
    return (q[:, q0:q1].contiguous(), kv_pool[..., k0:k1, :].contiguous(), q1 - q0, k1 - k0)


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
