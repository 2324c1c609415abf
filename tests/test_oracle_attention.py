"""Pins for the fp64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a library
routine (torch SDPA / logsumexp in fp64), a closed form, an invariant of
softmax attention, or an independent numpy statement of the split-KV merge.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A


def _f64(bits):
    return torch.from_numpy(W.bf16_bits_to_fp32(bits).astype(np.float64))


def _sdpa_reference(w):
    """Per request: contiguous K/V gathered with torch indexing, GQA by
    repeat_interleave, bottom-right causal mask, then torch SDPA in fp64."""
    outs, lses = [], []
    Hq, Hkv, T = w.num_q_heads, w.num_kv_heads, w.q_tokens
    G = Hq // Hkv
    kp = _f64(w.k_pages)
    vp = kp[..., :w.head_dim_v] if w.mla else _f64(w.v_pages)
    q = _f64(w.q)
    for b in range(w.batch):
        L = int(w.seqlens[b])
        pages = torch.from_numpy(w.page_table[b, :(L + w.page_size - 1) // w.page_size].astype(np.int64))
        k = kp[pages].reshape(-1, Hkv, w.head_dim_qk)[:L]          # [L][Hkv][Dk]
        v = vp[pages].reshape(-1, Hkv, w.head_dim_v)[:L]
        k = k.permute(1, 0, 2).repeat_interleave(G, dim=0)          # [Hq][L][Dk]
        v = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qb = q[b].permute(1, 0, 2)                                  # [Hq][T][Dk]
        if w.causal:
            mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]
        else:
            mask = torch.ones(T, L, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(qb, k, v, attn_mask=mask, scale=w.scale)
        s = w.scale * qb @ k.transpose(-1, -2)
        s = s.masked_fill(~mask, -math.inf)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(s, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


CASES = [
    dict(seqlens=[37, 200], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, page_size=16),
    dict(seqlens=[1, 5, 16, 17, 33], num_q_heads=4, num_kv_heads=4, head_dim_qk=32, page_size=16),
    dict(seqlens=[40, 9], q_tokens=4, num_q_heads=6, num_kv_heads=2, head_dim_qk=16, page_size=8),
    dict(seqlens=[70, 3], q_tokens=3, causal=False, num_q_heads=4, num_kv_heads=1,
         head_dim_qk=24, head_dim_v=40, page_size=4),
    dict(seqlens=[90, 31, 64], mla=True, num_q_heads=4, head_dim_qk=36, head_dim_v=32,
         page_size=16),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("seed", [0, 1])
def test_matches_torch_sdpa_fp64(case, seed):
    w = W.make_custom(seed=seed, **case)
    out, lse = A.decode_workload(w)
    ro, rl = _sdpa_reference(w)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_tiny_named_workload_matches_sdpa():
    w = W.make("tiny_gqa")
    out, lse = A.decode_workload(w)
    ro, rl = _sdpa_reference(w)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_length_one_returns_v0_and_its_score():
    w = W.make_custom([1, 1, 1], num_q_heads=4, num_kv_heads=2, head_dim_qk=16, seed=3)
    out, lse = A.decode_workload(w)
    for b in range(3):
        pg = w.page_table[b, 0]
        for h in range(4):
            g = h // 2
            v0 = W.bf16_bits_to_fp32(w.v_pages[pg, 0, g]).astype(np.float64)
            k0 = W.bf16_bits_to_fp32(w.k_pages[pg, 0, g]).astype(np.float64)
            q = W.bf16_bits_to_fp32(w.q[b, 0, h]).astype(np.float64)
            assert np.array_equal(out[b, 0, h], v0)
            assert lse[b, 0, h] == pytest.approx(w.scale * float(q @ k0), abs=1e-12)


@pytest.mark.parametrize("c", [1.5, -0.75, 2.0])
def test_constant_v_returns_the_constant(c):
    w = W.make_custom([3, 50, 129], num_q_heads=8, num_kv_heads=2, head_dim_qk=32, seed=4)
    w.v_pages[...] = W.fp32_to_bf16_bits(np.full(w.v_pages.shape, c, np.float32))
    out, _ = A.decode_workload(w)
    np.testing.assert_allclose(out, c, rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    w = W.make_custom([7, 100], q_tokens=2, num_q_heads=4, num_kv_heads=2, head_dim_qk=32, seed=5)
    w.v_pages[...] = W.fp32_to_bf16_bits(np.ones(w.v_pages.shape, np.float32))
    out, _ = A.decode_workload(w)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


def test_zero_keys_give_mean_of_values_and_log_n():
    w = W.make_custom([5, 64, 77], q_tokens=3, num_q_heads=4, num_kv_heads=2, head_dim_qk=16, seed=6)
    w.k_pages[...] = 0
    out, lse = A.decode_workload(w)
    for b in range(w.batch):
        L = int(w.seqlens[b])
        for t in range(3):
            n = L - 3 + t + 1
            for h in range(4):
                _, v = A.gather_rows(w, b, h // 2, n)
                np.testing.assert_allclose(out[b, t, h], v.mean(axis=0), rtol=0, atol=1e-12)
                assert lse[b, t, h] == pytest.approx(math.log(n), abs=1e-12)


def test_dominating_key_returns_its_value_row():
    w = W.make_custom([48], num_q_heads=2, num_kv_heads=1, head_dim_qk=16, seed=7)
    # q = e_0 for every head; key 29 gets +64 in dim 0, the rest are zero
    w.q[...] = 0
    w.q[..., 0] = W.fp32_to_bf16_bits(np.float32([1.0]))[0]
    w.k_pages[...] = 0
    pg, s = w.page_table[0, 29 // 16], 29 % 16
    w.k_pages[pg, s, 0, 0] = W.fp32_to_bf16_bits(np.float32([64.0]))[0]
    out, lse = A.decode_workload(w)
    v29 = W.bf16_bits_to_fp32(w.v_pages[pg, s, 0]).astype(np.float64)
    # weight of the other 47 keys is 47 e^{-64*scale}; with scale 1/4 that is 47 e^-16
    np.testing.assert_allclose(out[0, 0, 0], v29, rtol=0, atol=1e-4)
    assert lse[0, 0, 0] == pytest.approx(16.0 + math.log1p(47 * math.exp(-16.0)), abs=1e-12)


def test_causal_row_equals_single_token_on_shorter_prefix():
    T = 4
    w = W.make_custom([37, 64, 90], q_tokens=T, num_q_heads=4, num_kv_heads=2, head_dim_qk=32, seed=8)
    out, lse = A.decode_workload(w)
    for t in range(T):
        w1 = W.make_custom([37, 64, 90], q_tokens=1, num_q_heads=4, num_kv_heads=2,
                           head_dim_qk=32, seed=8)
        w1.k_pages, w1.v_pages, w1.page_table = w.k_pages, w.v_pages, w.page_table
        w1.q = np.ascontiguousarray(w.q[:, t:t + 1])
        w1.seqlens = (w.seqlens - T + t + 1).astype(np.int32)
        o1, l1 = A.decode_workload(w1)
        np.testing.assert_array_equal(out[:, t], o1[:, 0])
        np.testing.assert_array_equal(lse[:, t], l1[:, 0])


def test_page_permutation_invariance():
    w = W.make_custom([45, 130, 16], num_q_heads=8, num_kv_heads=2, head_dim_qk=32, seed=9,
                      spare_pages=3)
    out, lse = A.decode_workload(w)
    rng = np.random.default_rng(123)
    perm = rng.permutation(w.num_pages)          # new physical slot of old page p
    k2 = np.empty_like(w.k_pages)
    v2 = np.empty_like(w.v_pages)
    k2[perm] = w.k_pages
    v2[perm] = w.v_pages
    t2 = np.where(w.page_table >= 0, perm[np.maximum(w.page_table, 0)], -1).astype(np.int32)
    w.k_pages, w.v_pages, w.page_table = k2, v2, t2
    o2, l2 = A.decode_workload(w)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse, l2)


@pytest.mark.parametrize("seed", range(4))
def test_merge_of_any_partition_equals_unsplit(seed):
    rng = np.random.default_rng(seed)
    w = W.make_custom([int(rng.integers(2, 300))], q_tokens=1, num_q_heads=2, num_kv_heads=1,
                      head_dim_qk=32, head_dim_v=24, seed=seed)
    out, lse = A.decode_workload(w)
    L = int(w.seqlens[0])
    k, v = A.gather_rows(w, 0, 0, L)
    for h in range(2):
        q = W.bf16_bits_to_fp32(w.q[0, 0, h]).astype(np.float64)
        cuts = np.sort(rng.choice(np.arange(1, L), size=min(L - 1, int(rng.integers(1, 7))),
                                  replace=False)) if L > 1 else np.array([], int)
        edges = [0, *cuts.tolist(), L]
        parts = [A.partial_state(q, k[a:e], v[a:e], w.scale) for a, e in zip(edges[:-1], edges[1:])]
        parts.append(A.partial_state(q, k[:0], v[:0], w.scale))      # an empty split
        o, l = A.merge_states(parts)
        np.testing.assert_allclose(o, out[0, 0, h], rtol=0, atol=1e-12)
        assert l == pytest.approx(lse[0, 0, h], abs=1e-12)
        # lse of a two-way split is logaddexp of the two parts' lse
        mid = L // 2
        la = A.merge_states([A.partial_state(q, k[:mid], v[:mid], w.scale)])[1]
        lb = A.merge_states([A.partial_state(q, k[mid:], v[mid:], w.scale)])[1]
        assert np.logaddexp(la, lb) == pytest.approx(lse[0, 0, h], abs=1e-12)


def test_empty_request_gives_zero_and_minus_inf():
    w = W.make_custom([0, 20], q_tokens=2, num_q_heads=4, num_kv_heads=2, head_dim_qk=16, seed=10)
    out, lse = A.decode_workload(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_row_subset_matches_full():
    w = W.make_custom([33, 71], q_tokens=2, num_q_heads=4, num_kv_heads=2, head_dim_qk=16, seed=11)
    out, lse = A.decode_workload(w)
    rows = [0, 5, 9, 15]
    o, l = A.decode_workload(w, rows=rows)
    np.testing.assert_array_equal(o, out.reshape(-1, w.head_dim_v)[rows])
    np.testing.assert_array_equal(l, lse.reshape(-1)[rows])


def test_bad_inputs_are_rejected():
    w = W.make_custom([20, 40], num_q_heads=2, num_kv_heads=1, head_dim_qk=16, seed=12)
    bad = w.page_table.copy()
    bad[1, 1] = w.num_pages
    with pytest.raises(A.OracleInputError, match="page id"):
        A.decode(q=w.q, k_pages=w.k_pages, v_pages=w.v_pages, page_table=bad, seqlens=w.seqlens,
                 num_q_heads=2, num_kv_heads=1, head_dim_qk=16, head_dim_v=16, page_size=16,
                 causal=False, scale=0.25)
    with pytest.raises(A.OracleInputError, match="seqlen"):
        A.decode(q=w.q, k_pages=w.k_pages, v_pages=w.v_pages, page_table=w.page_table,
                 seqlens=np.array([20, 10_000], np.int32), num_q_heads=2, num_kv_heads=1,
                 head_dim_qk=16, head_dim_v=16, page_size=16, causal=False, scale=0.25)
    w2 = W.make_custom([3, 40], q_tokens=4, num_q_heads=2, num_kv_heads=1, head_dim_qk=16, seed=12)
    with pytest.raises(A.OracleInputError, match="causal"):
        A.decode_workload(w2)


def test_planted_mistakes_are_caught():
    """Plausible mistakes planted in a copy of the inputs' interpretation must
    move the result well beyond the GPU tolerance (so the pins have teeth)."""
    w = W.make_custom([37, 200], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, seed=0)
    ro, rl = _sdpa_reference(w)
    # interleaved instead of contiguous head grouping
    q2 = w.q.reshape(w.batch, 1, 4, 2, 64).transpose(0, 1, 3, 2, 4).reshape(w.q.shape)
    w2 = W.make_custom([37, 200], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, seed=0)
    w2.q = np.ascontiguousarray(q2)
    o2, _ = A.decode_workload(w2)
    assert np.abs(o2 - ro).max() > 0.1
    # off-by-one page mapping
    w3 = W.make_custom([37, 200], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, seed=0)
    w3.page_table = np.roll(w3.page_table, 1, axis=1)
    w3.page_table[w3.page_table < 0] = 0
    o3, _ = A.decode_workload(w3)
    assert np.abs(o3 - ro).max() > 0.1
