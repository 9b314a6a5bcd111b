"""Multi-rank host logic on CPU (gloo, world size 2): batch partition and the
max-over-ranks timing reduction used by the benchmark."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_flashattention_varlen_gb300 import dist as pdist


def test_partition_covers_every_sequence_once_and_balances():
    rng = np.random.default_rng(0)
    costs = rng.integers(1024, 8193, size=64).tolist()
    for world in (1, 2, 3, 8):
        parts = pdist.partition_by_cost(costs, world)
        flat = sorted(i for p in parts for i in p)
        assert flat == list(range(64))
        loads = [sum(costs[i] for i in p) for p in parts]
        assert max(loads) - min(loads) <= max(costs)
    assert pdist.partition_by_cost([], 2) == [[], []]
    with pytest.raises(ValueError):
        pdist.partition_by_cost([1], 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, costs, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = pdist.rank_world()
        mine = pdist.partition_by_cost(costs, w)[r]
        got = [None] * w
        dist.all_gather_object(got, mine)
        pdist.barrier()
        m = pdist.max_over_ranks(float(10 + r))
        q.put((r, got, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_partition_and_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    costs = [5, 9, 1, 7, 3, 3, 8]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, costs, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    parts = res[0][1]
    assert res[1][1] == parts
    assert sorted(i for p in parts for i in p) == list(range(len(costs)))
    assert set(parts[0]).isdisjoint(parts[1])
    assert res[0][2] == res[1][2] == 11.0
