"""The seeded input generator: deterministic, the stated shapes, NaN outside live rows."""
import numpy as np
import torch

import workloads


def test_named_tiny_decode_shapes():
    wl = workloads.named(1)
    assert list(wl.q.shape) == [16, 24, 256]
    assert list(wl.kv_pool.shape) == [22, 2, 64, 4, 256]
    assert list(wl.block_table.shape) == [2, 11]
    assert wl.cu_q.tolist() == [0, 8, 16] and wl.seq_lens.tolist() == [300, 650]
    bt = wl.block_table.numpy()
    assert (bt[0, :5] >= 0).all() and (bt[0, 5:] == -1).all() and (bt[1] >= 0).all()
    used = np.concatenate([bt[0, :5], bt[1]])
    assert len(set(used.tolist())) == 16
    assert wl.scale == 1.0 / 16 and wl.causal


def test_generator_is_deterministic():
    a = workloads.named(2, scale_down=16)
    b = workloads.named(2, scale_down=16)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.kv_pool.view(torch.int16), b.kv_pool.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)


def test_nan_fill_marks_dead_rows_only():
    wl = workloads.make_paged("t", 3, [2, 1], [70, 64], 4, 2, 16, 64, extra_pages=2)
    f = wl.kv_pool.float()
    bt = wl.block_table.numpy()
    # sequence 0 uses pages bt[0,0] (full) and bt[0,1] (6 live rows)
    assert torch.isfinite(f[bt[0, 0]]).all()
    assert torch.isfinite(f[bt[0, 1], :, :6]).all() and torch.isnan(f[bt[0, 1], :, 6:]).all()
    live = set(bt[bt >= 0].tolist())
    for p in range(wl.num_pages):
        if p not in live:
            assert torch.isnan(f[p]).all()


def test_full_size_workload_structure_without_drawing():
    # the decode batch: 64 sequences of one query, KV uniform in [1024, 8192]
    rng = np.random.default_rng(workloads.seed_for(2) + 100)
    lens = rng.integers(1024, 8192 + 1, size=64)
    assert lens.min() >= 1024 and lens.max() <= 8192


def test_visible_pairs_counts_the_causal_triangle():
    wl = workloads.make_paged("t", 4, [3], [5], 1, 1, 16, 64)
    assert wl.visible_pairs() == 3 + 4 + 5
    wl.causal = False
    assert wl.visible_pairs() == 15
