"""Host-side checks of libskdecode.so (no GPU needed): every symbol the header
declares is exported, the host planner equals the Stream-K definition in the
oracle bit for bit, and argument validation rejects bad calls before any CUDA
work is enqueued."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W
from oracle import streamk as S
from tests import plan_decode as PD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def N():
    from sm_load_balancing_gb300 import build as B
    B.build()
    from sm_load_balancing_gb300 import _native
    _native.lib()
    return _native


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(skd_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(N):
    lib = N.lib()
    declared = _declared_functions()
    assert declared, "no declarations found"
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(N.SIGNATURES), declared ^ set(N.SIGNATURES)
    assert lib.skd_abi_version() == 1


def _host_plan(N, seqlens, hkv, n, mode=0, page_size=16, seg_cost=None, align=None):
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    nb = N.lib().skd_plan_bytes(len(sl), hkv, n)
    buf = np.zeros(nb // 4, dtype=np.int32)
    if align is not None:
        st = N.lib().skd_decode_plan_aligned(sl.ctypes.data, len(sl), hkv, page_size, n, seg_cost or 0, align,
                                             buf.ctypes.data, nb)
    elif seg_cost is None:
        st = N.lib().skd_decode_plan(sl.ctypes.data, len(sl), hkv, page_size, n, mode, buf.ctypes.data, nb)
    else:
        st = N.lib().skd_decode_plan_weighted(sl.ctypes.data, len(sl), hkv, page_size, n, seg_cost,
                                              buf.ctypes.data, nb)
    return st, buf


def head_groups(hkv):
    """kv-head groups per request: heads go together in groups of the largest
    divisor of hkv not above 8 (the rule include/skdecode.h states)."""
    hg = max(g for g in range(1, min(hkv, 8) + 1) if hkv % g == 0)
    return hkv // hg


def _check_against_oracle(N, seqlens, hkv, n, seg_cost=None, align=None):
    st, buf = _host_plan(N, seqlens, hkv, n, seg_cost=seg_cost, align=align)
    assert st == 0
    p = PD.decode(buf)
    # an aligned plan is the split over cut units of 16 * align tokens, each
    # item's fixed cost rounded up to whole units
    a = align or 1
    ref = S.streamk_split(seqlens, head_groups(hkv), n, granule=16 * a, seg_cost=-(-(seg_cost or 0) // a))
    assert buf[13] == a  # the header records the cut unit
    got = [[(i, tb, te) for i, tb, te, _ in segs] for segs in p["segments"]]
    assert got == ref["segments"]
    assert p["total"] == ref["total_granules"]
    # slots: items with k > 1 splits own k consecutive slots, numbered in item order
    nxt = 0
    for i, splits in enumerate(ref["item_splits"]):
        assert p["nsplit"][i] == len(splits)
        if len(splits) > 1:
            assert p["slot0"][i] == nxt
            nxt += len(splits)
        else:
            assert p["slot0"][i] == -1
    assert p["nslots"] == nxt <= 2 * n
    for segs in p["segments"]:
        for i, tb, te, slot in segs:
            if p["nsplit"][i] == 1:
                assert slot == -1
            else:
                k = [x[1] for x in ref["item_splits"][i]].index(tb)
                assert slot == p["slot0"][i] + k
    assert p["nseg"] <= p["cap"]
    return p


@pytest.mark.parametrize("seed", range(40))
def test_host_planner_equals_streamk_definition(N, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(0, 9))
    hkv = int(rng.choice([1, 2, 3, 4, 8, 9, 10, 12, 16, 24, 32]))
    n = int(rng.choice([1, 2, 3, 7, 13, 148, 152, 304]))
    seqlens = [int(x) for x in rng.integers(0, 400, size=B)]
    if B and seed % 3 == 0:
        seqlens[int(rng.integers(0, B))] = 0
    _check_against_oracle(N, seqlens, hkv, n)


@pytest.mark.parametrize("name", ["tiny_gqa", "llama3_8b_gqa", "skewed_gqa", "mla_absorbed",
                                  "speculative_gqa"])
@pytest.mark.parametrize("n", [148, 152])
def test_host_planner_on_named_workloads(N, name, n):
    sl = W.draw_seqlens(name)
    hkv = {"tiny_gqa": 2, "mla_absorbed": 1}.get(name, 8)
    p = _check_against_oracle(N, sl.tolist(), hkv, n)
    per = [sum(-(-(te - tb) // 16) for _, tb, te, _ in segs) for segs in p["segments"]]
    assert max(per) - min(per) <= 1


@pytest.mark.parametrize("seed", range(24))
def test_weighted_planner_equals_definition(N, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 12))
    hkv = int(rng.choice([1, 2, 8, 12]))
    n = int(rng.choice([1, 2, 5, 13, 76, 148]))
    seg_cost = int(rng.choice([0, 1, 7, 40, 1000]))
    seqlens = [int(x) for x in rng.integers(0, 3000, size=B)]
    if seed % 4 == 0:
        seqlens[int(rng.integers(0, B))] = 0
    p = _check_against_oracle(N, seqlens, hkv, n, seg_cost=seg_cost)
    assert p["total"] == sum(head_groups(hkv) * (-(-L // 16) + (seg_cost if L else 0)) for L in seqlens)
    # every token granule is planned exactly once
    for i in range(len(seqlens) * head_groups(hkv)):
        L = seqlens[i // head_groups(hkv)]
        pieces = sorted((tb, te) for segs in p["segments"] for it, tb, te, _ in segs if it == i)
        if L == 0:
            assert pieces == [(0, 0)]
        else:
            assert pieces[0][0] == 0 and pieces[-1][1] == L
            assert all(a[1] == b[0] for a, b in zip(pieces, pieces[1:]))


def test_weighted_planner_zero_cost_is_plain_split(N):
    sl = W.draw_seqlens("mla_absorbed").tolist()
    _, a = _host_plan(N, sl, 1, 76)
    _, b = _host_plan(N, sl, 1, 76, seg_cost=0)
    assert np.array_equal(a, b)


def test_weighted_planner_gives_fewer_tokens_to_boundary_heavy_ctas(N):
    # one CTA range crosses many short requests: the cost moves tokens away from it
    sl = [4096] * 3 + [64] * 40 + [4096] * 3
    st, buf = _host_plan(N, sl, 1, 8, seg_cost=32)
    assert st == 0
    p = PD.decode(buf)
    toks = [sum(te - tb for _, tb, te, _ in segs) for segs in p["segments"]]
    nseg = [len(segs) for segs in p["segments"]]
    heavy = int(np.argmax(nseg))
    assert nseg[heavy] > 10 and toks[heavy] < min(t for c, t in enumerate(toks) if nseg[c] <= 2)
    assert _host_plan(N, sl, 1, 8, seg_cost=-1)[0] == N.SKD_EINVAL
    assert _host_plan(N, sl, 1, 8, seg_cost=70000)[0] == N.SKD_EINVAL


@pytest.mark.parametrize("seed", range(24))
def test_aligned_planner_equals_definition(N, seed):
    rng = np.random.default_rng(500 + seed)
    B = int(rng.integers(1, 12))
    hkv = int(rng.choice([1, 2, 8, 12]))
    n = int(rng.choice([1, 2, 5, 13, 76, 148]))
    seg_cost = int(rng.choice([0, 1, 8, 40, 1000]))
    align = int(rng.choice([1, 2, 3, 4, 64]))
    seqlens = [int(x) for x in rng.integers(0, 3000, size=B)]
    if seed % 4 == 0:
        seqlens[int(rng.integers(0, B))] = 0
    p = _check_against_oracle(N, seqlens, hkv, n, seg_cost=seg_cost, align=align)
    unit = 16 * align
    # every split point inside an item is a multiple of the unit; the pieces tile the item
    for i in range(len(seqlens) * head_groups(hkv)):
        L = seqlens[i // head_groups(hkv)]
        pieces = sorted((tb, te) for segs in p["segments"] for it, tb, te, _ in segs if it == i)
        if L == 0:
            assert pieces == [(0, 0)]
            continue
        assert pieces[0][0] == 0 and pieces[-1][1] == L
        assert all(a_[1] == b_[0] and a_[1] % unit == 0 for a_, b_ in zip(pieces, pieces[1:]))


def test_aligned_planner_one_is_weighted_plan(N):
    sl = W.draw_seqlens("mla_absorbed").tolist()
    for c in (0, 8, 40):
        _, a = _host_plan(N, sl, 1, 76, seg_cost=c)
        _, b = _host_plan(N, sl, 1, 76, seg_cost=c, align=1)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n", [76, 152])
def test_aligned_planner_reads_no_block_twice(N, n):
    # 64-token blocks (align 4): the blocks the CTAs touch add up to the blocks of
    # the batch, and with no segment cost the CTAs' block counts differ by at most one
    sl = W.draw_seqlens("mla_absorbed").tolist()
    st, buf = _host_plan(N, sl, 1, n, seg_cost=0, align=4)
    assert st == 0
    p = PD.decode(buf)
    per = [sum((te + 63) // 64 - tb // 64 for _, tb, te, _ in segs) for segs in p["segments"]]
    assert sum(per) == sum((L + 63) // 64 for L in sl)
    assert max(per) - min(per) <= 1
    assert _host_plan(N, sl, 1, n, seg_cost=0, align=0)[0] == N.SKD_EINVAL
    assert _host_plan(N, sl, 1, n, seg_cost=0, align=65)[0] == N.SKD_EINVAL


def test_head_group_rule():
    assert [head_groups(h) for h in [1, 2, 4, 7, 8, 9, 12, 16, 32]] == [1, 1, 1, 1, 1, 3, 2, 2, 4]


def test_round_robin_mode_matches_definition(N):
    seqlens = [5, 0, 9, 100, 33]
    st, buf = _host_plan(N, seqlens, 16, 4, mode=1)   # 16 kv heads -> 2 groups of 8
    assert st == 0
    p = PD.decode(buf)
    ref = S.round_robin_split(seqlens, 2, 4)
    assert [[s[:3] for s in segs] for segs in p["segments"]] == ref["segments"]
    assert p["nslots"] == 0 and all(ns == 1 for ns in p["nsplit"])


@pytest.mark.parametrize("seed", range(12))
def test_fixed_split_mode_matches_definition(N, seed):
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 40))
    hkv = int(rng.choice([1, 8, 16]))
    n = int(rng.choice([1, 7, 76, 152]))
    seqlens = [int(x) for x in rng.integers(0, 5000, size=B)]
    if seed % 3 == 0:
        seqlens[0] = 0
    st, buf = _host_plan(N, seqlens, hkv, n, mode=2)
    assert st == 0
    p = PD.decode(buf)
    ref = S.fixed_split(seqlens, head_groups(hkv), n)
    assert [[s_[:3] for s_ in segs] for segs in p["segments"]] == ref["segments"]
    # splits of an item own consecutive slots in split order, numbered in item order
    nxt = 0
    for i, parts in enumerate(ref["item_splits"]):
        assert p["nsplit"][i] == len(parts)
        if len(parts) > 1:
            assert p["slot0"][i] == nxt
            got = sorted((tb, slot) for segs in p["segments"] for it, tb, te, slot in segs if it == i)
            assert [slot for _, slot in got] == list(range(nxt, nxt + len(parts)))
            nxt += len(parts)
        else:
            assert p["slot0"][i] == -1
    assert p["nslots"] == nxt <= 2 * n


def test_planner_errors(N):
    st, _ = _host_plan(N, [10, -1], 1, 4)
    assert st == N.SKD_EINVAL
    st, _ = _host_plan(N, [10, 20], 1, 4, page_size=8)
    assert st == N.SKD_EINVAL
    sl = np.array([10, 20], np.int32)
    buf = np.zeros(4, np.int32)
    assert N.lib().skd_decode_plan(sl.ctypes.data, 2, 1, 16, 4, 0, buf.ctypes.data, 16) == N.SKD_EPLAN
    assert N.lib().skd_plan_bytes(2, 0, 4) == 0


def _shape(N, **kw):
    d = dict(batch=2, q_tokens=1, num_q_heads=8, num_kv_heads=2, head_dim_qk=64, head_dim_v=64,
             page_size=16, max_pages_per_req=16, num_pages=16, v_row_stride=64, scale=0.125,
             causal=0, kind=0)
    d.update(kw)
    return N.Shape(**d)


def test_workspace_bytes(N):
    lib = N.lib()
    s = _shape(N)
    nb = lib.skd_workspace_bytes(ctypes.byref(s), 148)
    rows, hg = 4, 2
    head = -(-rows * 67 // 4) * 4
    group_counters = 512
    partials = group_counters + -(-(4 * 2 * 148) // 256) * 256
    assert nb == partials + 2 * 148 * head * hg * 4
    assert lib.skd_workspace_bytes(ctypes.byref(_shape(N, head_dim_qk=96, head_dim_v=96,
                                                       v_row_stride=96)), 148) == 0
    assert lib.skd_workspace_bytes(ctypes.byref(_shape(N, num_q_heads=64, num_kv_heads=2)), 8) == 0
    mla = _shape(N, num_q_heads=128, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
                 v_row_stride=576, kind=1, page_size=64)
    assert lib.skd_workspace_bytes(ctypes.byref(mla), 148) > 0


def test_decode_attention_rejects_bad_arguments_before_launch(N):
    lib = N.lib()
    fake = 1 << 20  # never dereferenced: validation fails first
    s = _shape(N)

    def call(shape, q=fake, ws_bytes=1 << 30, n=4, ws=fake):
        return lib.skd_decode_attention(ctypes.byref(shape), q, fake, fake, fake, fake, fake, n,
                                        ws, ws_bytes, fake, fake, None)

    assert call(s, q=fake + 2) == N.SKD_EINVAL                      # misaligned q
    assert call(s, q=0) == N.SKD_EINVAL                             # null
    assert call(s, n=0) == N.SKD_EINVAL
    assert call(s, ws_bytes=100) == N.SKD_ESIZE
    assert call(_shape(N, head_dim_qk=80, head_dim_v=80, v_row_stride=80)) == N.SKD_EUNSUPPORTED
    assert call(_shape(N, page_size=8)) == N.SKD_EUNSUPPORTED
    assert call(_shape(N, num_q_heads=7)) == N.SKD_EINVAL
    assert call(_shape(N, scale=float("nan"))) == N.SKD_EINVAL
    assert call(_shape(N, kind=5)) == N.SKD_EINVAL
    assert call(_shape(N, batch=0)) == N.SKD_OK                     # nothing to do
    assert lib.skd_status_string(N.SKD_ESIZE) == b"workspace too small"
