"""Pins for the sparse (top-k) attention oracle (CPU only).

The sparse oracle restricts the plain attention to the cache positions a
request lists. It is checked against torch SDPA over the listed rows gathered
with torch indexing, against the dense oracle when every position is listed,
against closed forms (a repeated key, an empty list) and against invariants.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A


def _sparse_case(seqlens, k, seed=0, **kw):
    w = W.make_custom(seqlens, seed=seed, **kw)
    return W.select_topk(w, k, seed=seed + 100)


def _sdpa_sparse(w):
    """Per request: the listed K/V rows gathered by torch indexing, GQA by
    repeat_interleave, then torch SDPA / logsumexp in fp64 (no mask)."""
    Hq, Hkv, T = w.num_q_heads, w.num_kv_heads, w.q_tokens
    G = Hq // Hkv
    kp = torch.from_numpy(W.bf16_bits_to_fp32(w.k_pages).astype(np.float64))
    vp = kp[..., :w.head_dim_v] if w.mla else torch.from_numpy(W.bf16_bits_to_fp32(w.v_pages).astype(np.float64))
    q = torch.from_numpy(W.bf16_bits_to_fp32(w.q).astype(np.float64))
    outs, lses = [], []
    for b in range(w.batch):
        n = int(w.topk_len[b])
        pos = torch.from_numpy(w.topk_idx[b, :n].astype(np.int64))
        pages = torch.from_numpy(w.page_table[b].astype(np.int64))[pos // w.page_size]
        k = kp[pages, pos % w.page_size]                      # [n][Hkv][Dk]
        v = vp[pages, pos % w.page_size]
        k = k.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq][n][Dk]
        v = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qb = q[b].permute(1, 0, 2)                           # [Hq][T][Dk]
        if n == 0:
            outs.append(np.zeros((T, Hq, w.head_dim_v)))
            lses.append(np.full((T, Hq), -np.inf))
            continue
        o = torch.nn.functional.scaled_dot_product_attention(qb, k, v, scale=w.scale)
        s = w.scale * qb @ k.transpose(-1, -2)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(s, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


CASES = [
    dict(seqlens=[90, 31, 64, 0], mla=True, num_q_heads=4, head_dim_qk=36, head_dim_v=32, page_size=16),
    dict(seqlens=[200, 7, 50], num_q_heads=8, num_kv_heads=2, head_dim_qk=32, page_size=8),
    dict(seqlens=[129, 64], q_tokens=2, causal=False, num_q_heads=4, num_kv_heads=1, head_dim_qk=16,
         head_dim_v=24, page_size=4),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("k", [1, 17, 64])
def test_sparse_matches_torch_sdpa_on_gathered_rows(case, k):
    w = _sparse_case(k=k, seed=case, **CASES[case])
    out, lse = A.decode_sparse_workload(w)
    ro, rl = _sdpa_sparse(w)
    assert np.abs(out - ro).max() <= 1e-12
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.abs(lse[fin] - rl[fin]).max() <= 1e-12
    assert np.all(lse[~fin] == -np.inf) and np.all(out[~fin] == 0.0)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_listing_every_position_in_order_equals_dense(case):
    w = W.make_custom(seed=case, **CASES[case])
    L = w.seqlens
    idx = np.zeros((w.batch, max(int(L.max()), 1)), np.int32)
    for b, n in enumerate(L):
        idx[b, :n] = np.arange(n)
    ws = W.dataclasses.replace(w, topk_idx=idx, topk_len=L.copy())
    so, sl = A.decode_sparse_workload(ws)
    do, dl = A.decode_workload(w)
    # same keys in the same order: the same arithmetic, bit for bit
    assert np.array_equal(so, do) and np.array_equal(sl, dl)


def test_repeated_position_counts_twice():
    w = W.make_custom([40], mla=True, num_q_heads=2, head_dim_qk=8, head_dim_v=8, page_size=16, seed=3)
    j = 21
    idx = np.array([[j, j]], np.int32)
    ws = W.dataclasses.replace(w, topk_idx=idx, topk_len=np.array([2], np.int32))
    out, lse = A.decode_sparse_workload(ws)
    k, v = A.gather_rows(w, 0, 0, 40)
    q = W.bf16_bits_to_fp32(w.q[0, 0]).astype(np.float64)
    for h in range(2):
        s = w.scale * float(q[h] @ k[j])
        assert abs(lse[0, 0, h] - (s + math.log(2.0))) <= 1e-12
        assert np.abs(out[0, 0, h] - v[j]).max() <= 1e-12


def test_order_of_the_list_does_not_matter():
    w = _sparse_case([300, 77], 50, seed=5, num_q_heads=4, num_kv_heads=2, head_dim_qk=16, page_size=16)
    o1, l1 = A.decode_sparse_workload(w)
    rng = np.random.default_rng(0)
    idx = w.topk_idx.copy()
    for b in range(w.batch):
        n = int(w.topk_len[b])
        idx[b, :n] = idx[b, rng.permutation(n)]
    o2, l2 = A.decode_sparse_workload(W.dataclasses.replace(w, topk_idx=idx))
    assert np.abs(o1 - o2).max() <= 1e-12 and np.abs(l1 - l2).max() <= 1e-12


def test_listed_subset_equals_merge_of_its_parts():
    # the selection split in two parts gives two partial states whose merge is the whole
    w = _sparse_case([500], 120, seed=9, mla=True, num_q_heads=3, head_dim_qk=20, head_dim_v=12, page_size=8)
    out, lse = A.decode_sparse_workload(w)
    k, v = A.gather_rows(w, 0, 0, 500)
    q = W.bf16_bits_to_fp32(w.q[0, 0]).astype(np.float64)
    sel = w.topk_idx[0, :120]
    for h in range(3):
        parts = [A.partial_state(q[h], k[sel[:45]], v[sel[:45]], w.scale),
                 A.partial_state(q[h], k[sel[45:]], v[sel[45:]], w.scale)]
        mo, ml = A.merge_states(parts)
        assert np.abs(out[0, 0, h] - mo).max() <= 1e-12 and abs(lse[0, 0, h] - ml) <= 1e-12


def test_bad_lists_are_rejected():
    w = _sparse_case([30, 10], 8, seed=1, num_q_heads=2, num_kv_heads=1, head_dim_qk=8, page_size=8)
    bad = w.topk_idx.copy()
    bad[1, 0] = 10  # position == seqlen
    with pytest.raises(A.OracleInputError, match="position"):
        A.decode_sparse_workload(W.dataclasses.replace(w, topk_idx=bad))
    bad[1, 0] = -1
    with pytest.raises(A.OracleInputError, match="position"):
        A.decode_sparse_workload(W.dataclasses.replace(w, topk_idx=bad))
    with pytest.raises(A.OracleInputError, match="topk_len"):
        A.decode_sparse_workload(W.dataclasses.replace(w, topk_len=np.array([9, 2], np.int32)))


def test_select_topk_draws_distinct_positions_in_range():
    w = W.make_custom([5, 3000, 2048, 0], num_q_heads=2, num_kv_heads=1, head_dim_qk=8, page_size=16, seed=2)
    s1 = W.select_topk(w, 2048)
    s2 = W.select_topk(w, 2048)
    assert np.array_equal(s1.topk_idx, s2.topk_idx)  # seeded
    assert list(s1.topk_len) == [5, 2048, 2048, 0]
    for b, L in enumerate(w.seqlens):
        sel = s1.topk_idx[b, :s1.topk_len[b]]
        assert len(set(sel.tolist())) == len(sel)
        assert np.all((sel >= 0) & (sel < L))
    # the cache itself is untouched by the selection
    assert np.array_equal(s1.k_pages, w.k_pages) and np.array_equal(s1.q, w.q)
