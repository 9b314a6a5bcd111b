"""Seeded synthetic inputs for paged-KV varlen attention.

This module only draws random numbers and lays them out in memory. It holds
none of the attention arithmetic, so both the float64 oracle and the CUDA
library can be fed from it without sharing any of the method.

Layouts (element order, innermost last):

* ``q``        bf16 ``[total_q, n_heads_q, head_dim]``; sequence ``b`` owns rows
  ``cu_q[b] .. cu_q[b+1]``.
* ``kv_pool``  paged: bf16 ``[num_pages, 2 (K, V), page_size, n_heads_kv, head_dim]``;
  contiguous (``block_table is None``): bf16 ``[2 (K, V), sum(L), n_heads_kv, head_dim]``
  with sequence ``b`` at rows ``sum(L[:b]) ..``.
* ``block_table`` int32 ``[num_seqs, ceil(max_kv / page_size)]``, -1 for slots a
  sequence does not use.

Recipe (the same for every workload): ``numpy.random.default_rng(seed)``
(PCG64). Values are standard normal float32 rounded to bf16 (round to nearest
even, through torch). The page pool is drawn in one piece, then the physical
page of every logical slot comes from ``rng.permutation(num_pages)``. Rows past
a sequence's length in its last page, and every page no sequence uses, are
overwritten with NaN, so that a kernel which reads them shows it.

The five named workloads follow the launch manifest of the paged decode
example (trtllm-gen decode.json: buffers ``q``, ``kv``, ``table``, ``seq``,
``cuq``), the SageAttention2 GB10 benchmark shape (37,810 tokens, 56 heads,
head dim 128) and the hybrid-model decode graph (16 query / 2 KV heads,
head dim 256, page 64).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = ["Workload", "make_paged", "make_contiguous", "named", "NAMES", "seed_for"]


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor                      # bf16 [total_q, hq, d]
    kv_pool: torch.Tensor                # bf16, paged or contiguous layout (see module doc)
    block_table: Optional[torch.Tensor]  # int32 [B, max_pages] or None (contiguous)
    seq_lens: torch.Tensor               # int32 [B]
    cu_q: torch.Tensor                   # int32 [B + 1]
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    page_size: int
    num_pages: int                       # paged: pool pages; contiguous: rows per K/V plane
    scale: float
    causal: bool
    max_q: int
    max_kv: int

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    def q_lens(self) -> np.ndarray:
        cu = self.cu_q.numpy().astype(np.int64)
        return cu[1:] - cu[:-1]

    def visible_pairs(self) -> int:
        """Number of (query token, key) pairs the mask admits, per query head."""
        total = 0
        for ql, L in zip(self.q_lens().tolist(), self.seq_lens.numpy().tolist()):
            if not self.causal:
                total += ql * L
                continue
            for i in range(ql):
                total += max(0, min(L, L - ql + i + 1))
        return total

    def kv_bytes(self) -> int:
        """Bytes of live K and V rows: each row once per KV head (unused tails excluded)."""
        L = int(self.seq_lens.numpy().astype(np.int64).sum())
        return 2 * L * self.n_heads_kv * self.head_dim * 2

    def qo_bytes(self) -> int:
        return 2 * self.total_q * self.n_heads_q * self.head_dim * 2


def seed_for(config_index: int) -> int:
    """Seed of the numbered workload (1-based, in the order of ``NAMES``)."""
    return 1000 + config_index


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _cu(lens: Sequence[int]) -> torch.Tensor:
    c = np.zeros(len(lens) + 1, dtype=np.int64)
    c[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return torch.from_numpy(c.astype(np.int32))


def make_paged(
    name: str,
    seed: int,
    q_lens: Sequence[int],
    kv_lens: Sequence[int],
    n_heads_q: int,
    n_heads_kv: int,
    head_dim: int,
    page_size: int = 64,
    scale: Optional[float] = None,
    causal: bool = True,
    extra_pages: int = 0,
    nan_fill: bool = True,
    k_offset_std: float = 0.0,
) -> Workload:
    """Paged workload: pool ``[num_pages, 2, P, Hkv, D]`` with a shuffled block table."""
    rng = np.random.default_rng(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    B = len(kv_lens)
    assert len(q_lens) == B
    P = page_size
    pages_per_seq = [(L + P - 1) // P for L in kv_lens]
    used = int(sum(pages_per_seq))
    num_pages = max(1, used + int(extra_pages))
    max_kv = max(kv_lens) if B else 0
    max_q = max(q_lens) if B else 0
    max_pages = max(1, (max_kv + P - 1) // P)
    total_q = int(sum(q_lens))

    qf = rng.standard_normal((total_q, n_heads_q, head_dim), dtype=np.float32)
    pool = rng.standard_normal((num_pages, 2, P, n_heads_kv, head_dim), dtype=np.float32)
    if k_offset_std:
        off = rng.normal(0.0, k_offset_std, size=(n_heads_kv, head_dim)).astype(np.float32)
        pool[:, 0] += off[None, None, :, :]
    perm = rng.permutation(num_pages)

    table = np.full((B, max_pages), -1, dtype=np.int32)
    live = np.zeros(num_pages, dtype=bool)
    tail_rows = []  # (page, first dead row)
    nxt = 0
    for b in range(B):
        for s in range(pages_per_seq[b]):
            pg = int(perm[nxt])
            nxt += 1
            table[b, s] = pg
            live[pg] = True
        r = kv_lens[b] % P
        if pages_per_seq[b] and r:
            tail_rows.append((int(table[b, pages_per_seq[b] - 1]), r))
    if nan_fill:
        pool[~live] = np.nan
        for pg, r in tail_rows:
            pool[pg, :, r:] = np.nan

    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Workload(
        name=name, q=_bf16(qf), kv_pool=_bf16(pool), block_table=torch.from_numpy(table),
        seq_lens=torch.tensor(kv_lens, dtype=torch.int32), cu_q=_cu(q_lens),
        n_heads_q=n_heads_q, n_heads_kv=n_heads_kv, head_dim=head_dim, page_size=P,
        num_pages=num_pages, scale=float(scale), causal=bool(causal), max_q=max_q, max_kv=max_kv,
    )


def make_contiguous(
    name: str,
    seed: int,
    q_lens: Sequence[int],
    kv_lens: Sequence[int],
    n_heads_q: int,
    n_heads_kv: int,
    head_dim: int,
    scale: Optional[float] = None,
    causal: bool = False,
    k_offset_std: float = 0.0,
    page_size: int = 64,
) -> Workload:
    """Unpaged workload: K and V planes ``[2, sum(L), Hkv, D]``, no block table."""
    rng = np.random.default_rng(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    total_q = int(sum(q_lens))
    rows = int(sum(kv_lens))
    qf = rng.standard_normal((total_q, n_heads_q, head_dim), dtype=np.float32)
    kv = rng.standard_normal((2, max(rows, 1), n_heads_kv, head_dim), dtype=np.float32)
    if k_offset_std:
        off = rng.normal(0.0, k_offset_std, size=(n_heads_kv, head_dim)).astype(np.float32)
        kv[0] += off[None, :, :]
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Workload(
        name=name, q=_bf16(qf), kv_pool=_bf16(kv), block_table=None,
        seq_lens=torch.tensor(kv_lens, dtype=torch.int32), cu_q=_cu(q_lens),
        n_heads_q=n_heads_q, n_heads_kv=n_heads_kv, head_dim=head_dim, page_size=page_size,
        num_pages=max(rows, 1), scale=float(scale), causal=bool(causal),
        max_q=max(q_lens) if q_lens else 0, max_kv=max(kv_lens) if kv_lens else 0,
    )


def new_kv_rows(wl: Workload, seed: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """Seeded K and V rows of the query tokens, bf16 ``[total_q, Hkv, D]`` each
    (standard normal, like the pool), for the cache write in front of attention."""
    rng = np.random.default_rng(seed)
    shape = (int(wl.q.shape[0]), wl.n_heads_kv, wl.head_dim)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    return _bf16(k), _bf16(v)


NAMES: List[str] = [
    "tiny_paged_decode_2x8q_h24kv4_d256",
    "decode_64x1q_h32kv8_d128_L1k-8k",
    "causal_prefill_4x8192_h32kv8_d128",
    "noncausal_contig_1x37810_h56_d128",
    "mixed_96dec_4x2048chunk_h16kv2_d256",
]


def named(index: int, scale_down: int = 1) -> Workload:
    """The numbered workload (1..5, in the order of ``NAMES``).

    ``scale_down`` > 1 divides the token counts (used only to build small
    cases of the same structure for tests; 1 gives the full sizes).
    """
    seed = seed_for(index)
    if index == 1:
        # Two sequences, KV 300 and 650, the last 8 tokens of each are the
        # queries; 24 query heads over 4 KV heads, head dim 256, 22 pages of 64.
        return make_paged(NAMES[0], seed, [8, 8], [300, 650], 24, 4, 256, 64,
                          scale=1.0 / 16, causal=True, extra_pages=22 - 16)
    if index == 2:
        rng = np.random.default_rng(seed + 100)
        lens = rng.integers(1024, 8192 + 1, size=64)
        lens = np.maximum(1, lens // scale_down)
        return make_paged(NAMES[1], seed, [1] * 64, lens.tolist(), 32, 8, 128, 64,
                          scale=1.0 / math.sqrt(128), causal=True, extra_pages=16)
    if index == 3:
        n = 8192 // scale_down
        return make_paged(NAMES[2], seed, [n] * 4, [n] * 4, 32, 8, 128, 64,
                          scale=1.0 / math.sqrt(128), causal=True)
    if index == 4:
        n = 37810 // scale_down
        return make_contiguous(NAMES[3], seed, [n], [n], 56, 56, 128,
                               scale=1.0 / math.sqrt(128), causal=False, k_offset_std=0.5)
    if index == 5:
        rng = np.random.default_rng(seed + 100)
        dec = np.exp(rng.uniform(math.log(512), math.log(32768), size=96)).astype(np.int64)
        dec = np.maximum(1, dec // scale_down)
        chunk_q = 2048 // scale_down
        chunk_kv = (4096 + 2048) // scale_down
        q_lens = [1] * 96 + [chunk_q] * 4
        kv_lens = dec.tolist() + [chunk_kv] * 4
        return make_paged(NAMES[4], seed, q_lens, kv_lens, 16, 2, 256, 64,
                          scale=1.0 / 16, causal=True, extra_pages=8)
    raise ValueError(f"unknown workload {index}")
