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


def test_head_shard_covers_every_head_once():
    for hq, hkv in ((32, 8), (24, 4), (56, 56), (16, 2), (12, 3)):
        for world in (1, 2, 3, 4, 8):
            if world > hkv:
                continue
            spans = [pdist.head_shard(hq, hkv, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[0][2] == 0
            assert spans[-1][1] == hq and spans[-1][3] == hkv
            for (a, b) in zip(spans, spans[1:]):
                assert a[1] == b[0] and a[3] == b[2]
            sizes = [s[3] - s[2] for s in spans]
            assert max(sizes) - min(sizes) <= 1
            g = hq // hkv
            for q0, q1, k0, k1 in spans:
                # every query head of the block reads a KV head of the block
                assert all(k0 <= h // g < k1 for h in range(q0, q1))
    with pytest.raises(ValueError):
        pdist.head_shard(10, 4, 2, 0)
    with pytest.raises(ValueError):
        pdist.head_shard(8, 2, 2, 2)


def _head_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import workloads
        wl = workloads.make_paged("heads", 17, [3, 40, 1], [90, 200, 300], 16, 4, 128, 64, causal=True)
        q_r, kv_r, hq_r, hkv_r = pdist.shard_heads(wl.q, wl.kv_pool, wl.n_heads_q, wl.n_heads_kv, world, rank)
        part = workloads.Workload(**{**wl.__dict__, "q": q_r, "kv_pool": kv_r, "n_heads_q": hq_r,
                                     "n_heads_kv": hkv_r})
        out_r, _ = oracle.forward_workload(part)
        got = [None] * world
        dist.all_gather_object(got, out_r)
        if rank == 0:
            full, _ = oracle.forward_workload(wl)
            q.put((rank, bool(np.array_equal(np.concatenate(got, axis=1), full))))
        else:
            q.put((rank, True))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_head_shards_reassemble_the_whole_output():
    # each rank computes its KV heads' block (here with the oracle, the same
    # per-rank call the GPU path makes on its slices); gathered along the heads
    # the blocks are the whole batch's output, bit for bit
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_head_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == (0, True) and res[1] == (1, True)
