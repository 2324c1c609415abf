"""Pins for the work-split definitions (CPU only): the pages' two worked
examples (tests/golden/) plus invariants and brute-force enumeration."""
import json
import os

import numpy as np
import pytest

from oracle import streamk as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_four_sm_timeline_from_the_waves_page():
    g = _golden("waves_4sm_8task_timeline.json")
    r = S.list_schedule(g["task_times_ms"], g["n_workers"])
    assert [list(t) for t in r["tasks"]] == g["expected"]["tasks"]
    assert r["makespan"] == g["expected"]["makespan_ms"]
    assert r["idle"] == g["expected"]["idle_ms_per_sm"]
    loads = S.streamk_loads(g["task_times_ms"], g["n_workers"])
    assert loads == g["one_wave_equal_split"]["per_sm_ms"]
    assert max(loads) == g["one_wave_equal_split"]["makespan_ms"]


def test_streamk_split_on_the_timeline_tasks():
    """The same 8 tasks as work items of one kv head (granule 1 ms): the one-wave
    split gives every SM exactly 155 units."""
    g = _golden("waves_4sm_8task_timeline.json")
    r = S.streamk_split(g["task_times_ms"], 1, 4, granule=1)
    per = [sum(te - tb for _, tb, te in segs) for segs in r["segments"]]
    assert per == [155, 155, 155, 155]


def test_megartp_round_robin_queue_fill():
    g = _golden("megartp_round_robin_queues.json")
    q = S.round_robin_queues(g["n_tasks"], g["n_queues"])
    valid = (q >= 0).sum(axis=1)
    assert list(q.shape) == g["expected"]["padded_shape"]
    assert int((valid == 5).sum()) == g["expected"]["queues_with_5"]
    assert int((valid == 4).sum()) == g["expected"]["queues_with_4"]
    assert int((q < 0).sum()) == g["expected"]["noop_slots"]
    assert sorted(q[q >= 0].tolist()) == list(range(g["n_tasks"]))


def _brute_force_split(seqlens, hkv, n, granule, seg_cost=0):
    """Enumerate every granule of every item, deal contiguous index ranges.
    With ``seg_cost``, each non-empty item's granules are preceded by that many
    placeholder entries that belong to no segment."""
    units = []
    for b, L in enumerate(seqlens):
        for h in range(hkv):
            if L > 0:
                units += [(None, None)] * seg_cost
            for u in range(-(-L // granule)):
                units.append((b * hkv + h, u))
    total = len(units)
    out = []
    for c in range(n):
        lo, hi = c * total // n, (c + 1) * total // n
        segs = {}
        for item, u in units[lo:hi]:
            if item is not None:
                segs.setdefault(item, []).append(u)
        row = []
        for item in sorted(segs):
            us = segs[item]
            L = seqlens[item // hkv]
            row.append((item, min(us) * granule, min((max(us) + 1) * granule, L)))
        out.append(row)
    return out


@pytest.mark.parametrize("seed", range(30))
def test_streamk_split_matches_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 7))
    hkv = int(rng.integers(1, 4))
    n = int(rng.integers(1, 12))
    granule = int(rng.choice([1, 4, 16, 64]))
    seqlens = [int(x) for x in rng.integers(0, 120 if granule < 64 else 700, size=B)]
    if seed % 5 == 0:
        seqlens[0] = 0
    r = S.streamk_split(seqlens, hkv, n, granule)
    bf = _brute_force_split(seqlens, hkv, n, granule)
    nonempty = [[s for s in segs if s[2] > s[1]] for segs in r["segments"]]
    assert nonempty == bf
    # every token of every item covered exactly once, splits in order
    for i, splits in enumerate(r["item_splits"]):
        L = seqlens[i // hkv]
        if L == 0:
            assert len(splits) == 1 and splits[0][1:] == (0, 0)
            continue
        edges = [(tb, te) for _, tb, te in splits]
        assert edges[0][0] == 0 and edges[-1][1] == L
        assert all(a[1] == b[0] for a, b in zip(edges, edges[1:]))
        ctas = [c for c, _, _ in splits]
        assert ctas == sorted(ctas) and len(set(ctas)) == len(ctas)
    # near-equal chunks: granule counts differ by at most one
    per = [sum(-(-(te - tb) // granule) if te > tb else 0 for _, tb, te in segs)
           for segs in r["segments"]]
    b = r["bounds"]
    assert per == [b[c + 1] - b[c] for c in range(n)]
    assert max(per) - min(per) <= 1
    nseg = sum(len(s) for s in r["segments"])
    assert nseg <= B * hkv + n - 1 + sum(1 for L in seqlens if L == 0) * hkv
    # segments of a CTA are in item order
    for segs in r["segments"]:
        items = [s[0] for s in segs]
        assert items == sorted(items)


@pytest.mark.parametrize("seed", range(30))
def test_weighted_split_matches_brute_force(seed):
    # the segment-cost extension and the coarse cut unit (granule 64 = the MLA
    # kernel's block): the same split as dealing placeholder entries + granules
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 7))
    hkv = int(rng.integers(1, 4))
    n = int(rng.integers(1, 12))
    granule = int(rng.choice([1, 16, 64]))
    seg_cost = int(rng.choice([0, 1, 3, 10]))
    seqlens = [int(x) for x in rng.integers(0, 300 if granule < 64 else 1500, size=B)]
    if seed % 4 == 0:
        seqlens[0] = 0
    r = S.streamk_split(seqlens, hkv, n, granule, seg_cost=seg_cost)
    bf = _brute_force_split(seqlens, hkv, n, granule, seg_cost=seg_cost)
    assert [[s for s in segs if s[2] > s[1]] for segs in r["segments"]] == bf
    assert r["total_granules"] == sum(hkv * (-(-L // granule) + (seg_cost if L else 0)) for L in seqlens)
    # split points fall on multiples of the granule
    for i, splits in enumerate(r["item_splits"]):
        assert all(tb % granule == 0 for _, tb, _ in splits)


def test_round_robin_split_deals_whole_items():
    r = S.round_robin_split([5, 0, 9], 2, 4)
    assert r["segments"] == [[(0, 0, 5), (4, 0, 9)], [(1, 0, 5), (5, 0, 9)], [(2, 0, 0)], [(3, 0, 0)]]


def test_fixed_split_hand_example():
    # 3 items on 7 CTAs: S = 7 // 3 = 2 splits per item. Item 0 has 7 granules
    # (100 tokens): granules [0, 3) and [3, 7) -> tokens [0, 48) and [48, 100);
    # item 1 is empty: one empty piece; item 2 has 3 granules: [0, 1), [1, 3) ->
    # tokens [0, 16), [16, 40). The five pieces go to CTAs 0..4 in that order.
    r = S.fixed_split([100, 0, 40], 1, 7)
    assert r["splits_per_item"] == 2
    assert r["item_splits"] == [[(0, 48), (48, 100)], [(0, 0)], [(0, 16), (16, 40)]]
    assert r["segments"] == [[(0, 0, 48)], [(0, 48, 100)], [(1, 0, 0)], [(2, 0, 16)], [(2, 16, 40)], [], []]


@pytest.mark.parametrize("seed", range(20))
def test_fixed_split_properties(seed):
    rng = np.random.default_rng(2000 + seed)
    B = int(rng.integers(1, 9))
    hkv = int(rng.integers(1, 4))
    n = int(rng.integers(1, 40))
    seqlens = [int(x) for x in rng.integers(0, 500, size=B)]
    r = S.fixed_split(seqlens, hkv, n)
    items = B * hkv
    assert r["splits_per_item"] == max(1, n // items)
    flat = []
    for i, parts in enumerate(r["item_splits"]):
        L = seqlens[i // hkv]
        g = -(-L // 16)
        assert len(parts) == max(1, min(r["splits_per_item"], g))
        assert parts[0][0] == 0 and parts[-1][1] == L
        assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
        if g:
            sizes = [-(-(te - tb) // 16) for tb, te in parts]  # granules per piece
            assert max(sizes) - min(sizes) <= 1 and sum(sizes) == g
            assert all(tb % 16 == 0 for tb, _ in parts)
        flat += [(i, tb, te) for tb, te in parts]
    # piece j of the (item, split) order goes to CTA j mod n
    for j, seg in enumerate(flat):
        assert seg in r["segments"][j % n]
    assert sum(len(s) for s in r["segments"]) == len(flat)
    if items <= n:
        assert all(len(s) <= 1 for s in r["segments"])
