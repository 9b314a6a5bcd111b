"""The tile plan, exactly: the device planner's two work lists (through
``pattn_plan_items``) against the tiling rules written out here on the host.

For every sequence, KV head and q tile the items must cover the visible KV
tiles [0, n) once, in contiguous ranges; only units of a single q tile are
split, into the balanced ranges [s n / S, (s + 1) n / S); a split unit's
partial rows are its own; units of at most 16 packed query rows go to the
decode kernel's list; each list is ordered longest first; q tiles that see no
key make no item; rejected sequences make none. Integer work: every check is
exact."""
import collections

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a GPU", allow_module_level=True)

BM, DEC_ROWS, DEC_BN, MAX_SPLITS, SEQ_BITS = 128, 16, 128, 64, 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_flashattention_varlen_gb300 import build
    build.build()


def cdiv(a, b):
    return -(-a // b)


def dec_possible(wl):
    """The decode kernel serves units of <= 16 packed rows, unless the bounds
    rule them out: every sequence holds >= total_q - (B - 1) * max_q queries."""
    G = wl.n_heads_q // wl.n_heads_kv
    min_ql = wl.total_q - (wl.num_seqs - 1) * max(wl.max_q, 0)
    return G <= DEC_ROWS and min_ql * G <= DEC_ROWS


def expected_units(wl, rejected=()):
    """(list, b, q tile) -> visible KV tiles, for every q tile that makes an item."""
    G = wl.n_heads_q // wl.n_heads_kv
    T = BM // G
    # two q tiles per item: CTA pairs at head_dim 256, two-q-tile CTAs at 128 (non-causal)
    pair = wl.max_q > T and (wl.head_dim == 256 or not wl.causal)
    bn_pre = 128 if (wl.head_dim == 128 or pair) else 64
    cu = wl.cu_q.numpy().astype(np.int64)
    sl = wl.seq_lens.numpy().astype(np.int64)
    units = {}
    for b in range(wl.num_seqs):
        ql, L = int(cu[b + 1] - cu[b]), int(sl[b])
        if ql <= 0 or b in rejected:
            continue
        dec = dec_possible(wl) and ql * G <= DEC_ROWS
        bn = DEC_BN if dec else bn_pre
        nqt = cdiv(ql, T)

        def tiles(qt):
            hi = min(L, L - ql + min(ql, (qt + 1) * T)) if wl.causal else L
            return cdiv(hi, bn) if hi > 0 else 0

        for qt in range(nqt):
            if pair and not dec:
                if qt & 1:
                    continue
                n = tiles(min(qt + 1, nqt - 1))
            else:
                n = tiles(qt)
            if n > 0:
                units[(1 if dec else 0, b, qt)] = (n, nqt, ql * G)
    return units


def check_plan(wl, rejected=()):
    import paged_kv_flashattention_varlen_gb300 as pk
    dev = torch.device("cuda:0")
    bt = None if wl.block_table is None else wl.block_table.to(dev)
    pre, dec, counts = pk.plan_items(bt, wl.seq_lens.to(dev), wl.cu_q.to(dev), total_q=int(wl.q.shape[0]),
                                     max_q=wl.max_q, max_kv=wl.max_kv, n_heads_q=wl.n_heads_q,
                                     n_heads_kv=wl.n_heads_kv, head_dim=wl.head_dim, causal=wl.causal,
                                     num_pages=wl.num_pages)
    assert counts[0] == len(pre) and counts[1] == len(dec)
    units = expected_units(wl, rejected)
    hkv = wl.n_heads_kv
    got = collections.defaultdict(list)  # (list, b, hk, qt) -> [(k0, k1, split, w)]
    for lst, items in ((0, pre), (1, dec)):
        cost = (items[:, 2] & 0xFFFF) - ((items[:, 2] >> 16) & 0xFFFF)
        assert np.all(cost > 0)
        assert np.all(np.diff(np.minimum(cost, 1023)) <= 0), "list not longest first"
        for x, y, z, w in items.tolist():
            b, s = x & ((1 << SEQ_BITS) - 1), x >> SEQ_BITS
            hk, qt = y >> 16, y & 0xFFFF
            assert 0 <= hk < hkv
            got[(lst, b, hk, qt)].append((z >> 16, z & 0xFFFF, s, w))
    want_keys = {(lst, b, hk, qt) for (lst, b, qt) in units for hk in range(hkv)}
    assert set(got) == want_keys, (sorted(set(got) ^ want_keys)[:8])
    split_units, part_ranges = 0, []
    for (lst, b, hk, qt), its in got.items():
        n, nqt, rows = units[(lst, b, qt)]
        its.sort()
        S = len(its)
        assert its[0][0] == 0 and its[-1][1] == n, "KV range not covered"
        for a, c in zip(its, its[1:]):
            assert a[1] == c[0], "gap or overlap between splits"
        if S == 1:
            assert its[0][2] == 0 and its[0][3] == -1
            continue
        assert nqt == 1 and S <= MAX_SPLITS, "only single-q-tile units split"
        for k0, k1, s, w in its:
            assert (k0, k1) == (s * n // S, (s + 1) * n // S), "unbalanced split"
        ss = sorted(i[2] for i in its)
        assert ss == list(range(S))
        part0 = {w - (hk * S + s) * rows for _, _, s, w in its}
        assert len(part0) == 1, "partial rows of one unit not in its slots"
        p0 = part0.pop()
        part_ranges.append((p0 + hk * S * rows, p0 + (hk + 1) * S * rows))
        split_units += 1
    assert split_units == counts[2]
    part_ranges.sort()
    for a, c in zip(part_ranges, part_ranges[1:]):
        assert a[1] <= c[0], "partial rows shared by two units"
    if part_ranges:
        assert part_ranges[0][0] >= 0 and part_ranges[-1][1] <= counts[3]
    return counts


@pytest.mark.parametrize("index,scale_down", [(1, 1), (2, 1), (3, 16), (4, 32), (5, 8), (5, 1)])
def test_named_workload_plans(index, scale_down):
    check_plan(workloads.named(index, scale_down=scale_down))


def test_decode_batch_splits_long_units():
    counts = check_plan(workloads.named(2))
    assert counts[2] > 0  # the longest decode units take the split-KV path


@pytest.mark.parametrize("d,hq,hkv", [(128, 4, 1), (128, 8, 8), (128, 32, 2), (256, 12, 2), (256, 16, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_edge_length_plans(d, hq, hkv, causal):
    edges = [1, 63, 64, 65, 127, 128, 129]
    q_lens, kv_lens = [], []
    for L in edges:
        for ql in edges:
            if causal and ql > L:
                continue
            q_lens.append(ql)
            kv_lens.append(L)
    check_plan(workloads.make_paged("plan_edges", 700 + d + hq, q_lens, kv_lens, hq, hkv, d, 64,
                                    causal=causal, extra_pages=1))


def test_empty_sequences_and_queries_before_the_first_key():
    check_plan(workloads.make_paged("plan_empty", 71, [3, 0, 5, 2, 40], [0, 10, 3, 70, 0], 8, 2, 128, 64,
                                    causal=False, extra_pages=1))


def test_rejected_sequence_makes_no_item():
    import paged_kv_flashattention_varlen_gb300 as pk
    wl = workloads.make_paged("plan_bad", 72, [2, 30, 1], [100, 300, 900], 8, 2, 128, 64, causal=True)
    wl.block_table[1, 2] = wl.num_pages + 5  # a live entry outside the pool
    check_plan(wl, rejected={1})
    assert pk.device_status() != 0  # reported on the error word (and cleared by the read)
    assert pk.device_status() == 0


def test_contiguous_cache_plan():
    check_plan(workloads.make_contiguous("plan_c", 73, [40, 1, 7, 300], [300, 129, 64, 300], 8, 2, 128,
                                         causal=True))


def host_decode_target_items(wl, sms):
    """The decode list's item count under the planner's split rule, written
    out on the host. Base target: 2 items per SM (at most 409). When the
    decode units' lengths are skewed (longest unit more than 2.5 times the
    mean), some unit exceeds the smallest split (8 tiles) and there are at
    most 4 units per CTA, the target is chosen between the base and a quarter
    more: each unit of T KV tiles split into min(ceil(T / chunk_tiles), 64, T)
    parts, item costs counting-sorted longest first (clamped at 1023), the
    decode kernel's alternating round robin over `sms` CTAs, each item costing
    its tiles + 2; the candidate with the smaller largest CTA load wins (ties:
    the base)."""
    G = wl.n_heads_q // wl.n_heads_kv
    hkv = wl.n_heads_kv
    cu = wl.cu_q.numpy().astype(np.int64)
    sl = wl.seq_lens.numpy().astype(np.int64)
    base = min(4 * sms // 2, 512 * 4 // 5)
    cands = [base, base + base // 4]
    tiles = []
    for b in range(wl.num_seqs):
        ql, L = int(cu[b + 1] - cu[b]), int(sl[b])
        if dec_possible(wl) and 1 <= ql and ql * G <= DEC_ROWS:
            tiles.append(cdiv(L, DEC_BN) if L > 0 else 0)
    work = sum(2 * t for t in tiles) * hkv
    units = len(tiles) * hkv

    def splits(t, target):
        chunk = max(cdiv(work, max(target, 1)), 16)
        ct = max(1, cdiv(chunk, 2))
        return min(cdiv(t, ct), MAX_SPLITS, t) if t >= 2 else 1

    def items(target):
        out = []
        for t in tiles:
            if t == 0:
                continue
            S = splits(t, target)
            out += [min((s + 1) * t // S - s * t // S, 1023) for s in range(S)] * hkv
        return sorted(out, reverse=True)

    def max_load(its):
        best = 0
        for c in range(sms):
            load, k, pos = 0, 0, c
            while pos < len(its):
                load += its[pos] + 2
                k += 1
                pos = (k + 1) * sms - 1 - c if k & 1 else k * sms + c
            best = max(best, load)
        return best

    tmax = max(tiles) if tiles else 0
    skewed = 4 * tmax * units > 5 * work
    choose = skewed and tmax > 8 and units <= 4 * sms
    target = base
    if choose and max_load(items(cands[1])) < max_load(items(cands[0])):
        target = cands[1]
    return len(items(target)), choose, target


def _random_decode_mix(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(8, 76))
    kv = np.exp(rng.uniform(np.log(64), np.log(40000), size=n)).astype(int).tolist()
    return workloads.make_paged("plan_dec_mix", 800 + seed, [1] * n, kv, 32, 8, 128, 64, causal=True,
                                nan_fill=False)


@pytest.mark.parametrize("case", ["decode_batch", "mixed", "mix0", "mix1", "mix2", "mix3"])
def test_decode_split_target_follows_the_balance_model(case):
    wl = {"decode_batch": lambda: workloads.named(2), "mixed": lambda: workloads.named(5),
          "mix0": lambda: _random_decode_mix(0), "mix1": lambda: _random_decode_mix(1),
          "mix2": lambda: _random_decode_mix(2), "mix3": lambda: _random_decode_mix(3)}[case]()
    counts = check_plan(wl)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_items, _, _ = host_decode_target_items(wl, sms)
    assert counts[1] == n_items
