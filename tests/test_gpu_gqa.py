"""GQA decode attention on the GPU against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests import plan_decode as PD
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev, compare

pytestmark = pytest.mark.gpu


def _check(w, **kw):
    d = Dev(w)
    out, lse, err, _ = d.run(**kw)
    assert err == 0
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
    return out, lse


def test_tiny_named_workload():
    _check(W.make("tiny_gqa"))


# several tiles, ragged tails, empty and one-token requests, T>1 causal, D=64/128
MEDIUM = [
    dict(seqlens=[1, 15, 16, 17, 63, 64, 65, 200, 1000, 0, 3000], num_q_heads=32, num_kv_heads=8,
         head_dim_qk=128, page_size=16),
    dict(seqlens=[700, 33, 4100, 0, 129], num_q_heads=64, num_kv_heads=8, head_dim_qk=128,
         page_size=64),
    dict(seqlens=[4, 5, 77, 2048, 999], q_tokens=4, num_q_heads=32, num_kv_heads=8,
         head_dim_qk=128, page_size=16),
    dict(seqlens=[37, 200, 5000, 1], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, page_size=16),
    dict(seqlens=[300, 2], q_tokens=2, num_q_heads=16, num_kv_heads=2, head_dim_qk=64,
         page_size=32),
    dict(seqlens=[513, 1024, 40], q_tokens=3, causal=False, num_q_heads=20, num_kv_heads=4,
         head_dim_qk=128, page_size=16),
    # kv heads in groups of 6 (two groups per request) and of 8 (two groups)
    dict(seqlens=[260, 1500, 31], num_q_heads=24, num_kv_heads=12, head_dim_qk=64, page_size=16),
    dict(seqlens=[900, 77, 2222], q_tokens=2, num_q_heads=32, num_kv_heads=16, head_dim_qk=128,
         page_size=32),
    dict(seqlens=[333, 64], num_q_heads=9, num_kv_heads=3, head_dim_qk=128, page_size=16),
]


@pytest.mark.parametrize("case", range(len(MEDIUM)))
@pytest.mark.parametrize("n_ctas", [1, 3, 7, None, 400])
def test_medium_cases_any_grid(case, n_ctas):
    _check(W.make_custom(seed=case, **MEDIUM[case]), n_ctas=n_ctas)


@pytest.mark.parametrize("case", [0, 2])
def test_round_robin_plan_gives_same_result(case):
    w = W.make_custom(seed=case, **MEDIUM[case])
    _check(w, mode="round_robin")


@pytest.mark.parametrize("case", range(len(MEDIUM)))
@pytest.mark.parametrize("n_ctas", [7, None])
def test_two_kernel_comparator_fixed_split(case, n_ctas):
    # fixed splits merged by the separate combine kernel ...
    w = W.make_custom(seed=case, **MEDIUM[case])
    _check(w, mode="fixed_split", n_ctas=n_ctas, two_kernel=True)


@pytest.mark.parametrize("case", [0, 2, 3])
def test_fixed_split_plan_with_just_in_time_merge(case):
    # ... and the same plan merged just in time by the one-kernel entry point
    w = W.make_custom(seed=case, **MEDIUM[case])
    _check(w, mode="fixed_split")


def test_result_independent_of_plan_and_repeatable():
    w = W.make_custom(seed=11, **MEDIUM[0])
    d = Dev(w)
    outs = {}
    for n in [1, 2, 5, 148, 152, 304]:
        o, l, err, _ = d.run(n_ctas=n)
        assert err == 0
        outs[n] = (o.float().cpu().numpy(), l.cpu().numpy())
    a = outs[152]
    for n, (o, l) in outs.items():
        assert np.abs(o - a[0]).max() <= OUT_TOL
        fin = np.isfinite(a[1])  # rows of empty requests have lse = -inf under every plan
        assert np.array_equal(np.isfinite(l), fin)
        assert np.abs(l[fin] - a[1][fin]).max(initial=0.0) <= LSE_TOL
    # same plan twice: identical bits (the merge order is fixed by split index)
    o1, l1, _, ws = d.run(n_ctas=152)
    o2, l2, _, _ = d.run(n_ctas=152, ws=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_page_permutation_is_bitwise_invariant():
    w = W.make_custom(seed=5, spare_pages=7, **MEDIUM[0])
    d = Dev(w)
    o1, l1, err, _ = d.run()
    assert err == 0
    perm = np.random.default_rng(9).permutation(w.num_pages)
    k2 = np.empty_like(w.k_pages)
    v2 = np.empty_like(w.v_pages)
    k2[perm] = w.k_pages
    v2[perm] = w.v_pages
    w.k_pages, w.v_pages = k2, v2
    w.page_table = np.where(w.page_table >= 0, perm[np.maximum(w.page_table, 0)], -1).astype(np.int32)
    o2, l2, err, _ = Dev(w).run()
    assert err == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_invariants_length_one_and_constant_v():
    w = W.make_custom([1, 1, 50, 333], num_q_heads=16, num_kv_heads=4, head_dim_qk=128, seed=3)
    w.v_pages[:, :, :, :] = W.fp32_to_bf16_bits(np.full(w.v_pages.shape, 1.5, np.float32))
    d = Dev(w)
    out, lse, err, _ = d.run()
    assert err == 0
    o = out.float().cpu().numpy()
    assert np.all(o == 1.5)          # constant V returns that constant (exactly, in bf16)
    ro, rl = A.decode_workload(w)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    # L = 1: the one value row comes back; lse is that key's score
    w2 = W.make_custom([1, 1], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, seed=4)
    out2, lse2, _, _ = Dev(w2).run()
    for b in range(2):
        pg = w2.page_table[b, 0]
        for h in range(8):
            v0 = W.bf16_bits_to_fp32(w2.v_pages[pg, 0, h // 4])
            assert np.array_equal(out2[b, 0, h].float().cpu().numpy(), v0)


def test_weights_sum_to_one_with_ones_v():
    w = W.make_custom([17, 4000, 123], q_tokens=4, num_q_heads=32, num_kv_heads=8,
                      head_dim_qk=128, seed=6)
    w.v_pages[...] = W.fp32_to_bf16_bits(np.ones(w.v_pages.shape, np.float32))
    out, _, err, _ = Dev(w).run()
    assert err == 0 and np.all(out.float().cpu().numpy() == 1.0)


def test_device_planner_matches_host_planner():
    import sm_load_balancing_gb300 as skd
    rng = np.random.default_rng(0)
    for trial in range(25):
        B = int(rng.integers(0, 70))
        hkv = int(rng.integers(1, 9))
        n = int(rng.choice([1, 3, 148, 152, 1000, 2000]))
        sl = rng.integers(0, 5000, size=B).astype(np.int32)
        if B and trial % 4 == 0:
            sl[rng.integers(0, B)] = 0
        host = skd.plan(sl, hkv, 16, n)
        dev = skd.plan_device(torch.from_numpy(sl).cuda(), hkv, 16, n)
        torch.cuda.synchronize()
        assert torch.equal(host, dev.cpu()), (trial, B, hkv, n)
    for name, hkv in [("skewed_gqa", 8), ("llama3_8b_gqa", 8), ("mla_absorbed", 1)]:
        sl = W.draw_seqlens(name)
        host = skd.plan(sl, hkv, 64, 152)
        dev = skd.plan_device(torch.from_numpy(sl).cuda(), hkv, 64, 152)
        assert torch.equal(host, dev.cpu())
    # the weighted split, same bytes on both sides
    for trial in range(12):
        B = int(rng.integers(1, 70))
        hkv = int(rng.choice([1, 2, 8]))
        n = int(rng.choice([1, 76, 152]))
        c = int(rng.choice([1, 40, 999]))
        al = int(rng.choice([1, 3, 4, 64]))
        sl = rng.integers(0, 9000, size=B).astype(np.int32)
        if trial % 3 == 0:
            sl[rng.integers(0, B)] = 0
        host = skd.plan(sl, hkv, 16, n, seg_cost=c, align=al)
        dev = skd.plan_device(torch.from_numpy(sl).cuda(), hkv, 16, n, seg_cost=c, align=al)
        torch.cuda.synchronize()
        assert torch.equal(host, dev.cpu()), (trial, B, hkv, n, c, al)


def test_device_plan_drives_the_kernel():
    import sm_load_balancing_gb300 as skd
    w = W.make_custom(seed=2, **MEDIUM[1])
    d = Dev(w)
    n = skd.sm_count()
    plan = skd.plan_device(d.sl, 8, w.page_size, n)
    out, lse, err, _ = d.run(n_ctas=n, plan=plan)
    assert err == 0
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL


def test_device_errors_are_reported_not_faulted():
    import sm_load_balancing_gb300 as skd
    w = W.make_custom([40, 100], num_q_heads=8, num_kv_heads=2, head_dim_qk=64, seed=1)
    d = Dev(w)
    # a page id outside the cache: the kernel substitutes page 0 and flags it
    bad = w.page_table.copy()
    bad[1, 2] = w.num_pages + 5
    d.pt = torch.from_numpy(bad).cuda()
    _, _, err, ws = d.run()
    assert err & skd.SKD_DEVERR_PAGE
    # a plan built for another grid size is rejected by the kernel
    d2 = Dev(w)
    n = skd.sm_count()
    wrong = skd.plan(w.seqlens, 2, 16, n + 1).cuda()
    ws2 = skd.workspace(d2.shape, n + 1)
    skd.decode_attention(d2.q, d2.k, d2.v, d2.pt, d2.sl, wrong, ws2, scale=w.scale, n_ctas=n,
                         shape=d2.shape)
    torch.cuda.synchronize()
    assert skd.read_error(ws2) & skd.SKD_DEVERR_PLAN
    # device seqlens longer than the plan's ranges are flagged
    d3 = Dev(w)
    plan = skd.plan(np.array([40, 100], np.int32), 2, 16, n).cuda()
    d3.sl = torch.tensor([40, 20], dtype=torch.int32, device="cuda")
    _, _, err3, _ = d3.run(n_ctas=n, plan=plan)
    assert err3 & skd.SKD_DEVERR_SEQLEN
    # after a reset the same workspace works again
    skd.read_error(ws)
    from sm_load_balancing_gb300 import _native as N
    N.lib().skd_workspace_reset(ws.data_ptr(), ws.numel(), None)
    out, lse, err4, _ = Dev(w).run(ws=ws)
    assert err4 == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama3_8b_gqa", "skewed_gqa", "speculative_gqa"])
def test_named_workload_full_size(name):
    """Full-size workloads in the launch configuration the benchmark times
    (one CTA per SM, Stream-K plan), every row against the oracle."""
    w = W.make(name)
    d = Dev(w)
    out, lse, err, _ = d.run()
    assert err == 0
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)


def test_skewed_long_request_first_and_last():
    """The long request at the first and at the last batch position (scaled
    down: one 40000-token request among 63 short ones)."""
    rng = np.random.default_rng(1)
    short = rng.integers(64, 1024, size=63).tolist()
    for seq in ([40000] + short, short + [40000]):
        w = W.make_custom(seq, num_q_heads=64, num_kv_heads=8, head_dim_qk=128, page_size=64, seed=2)
        _check(w)


@pytest.mark.parametrize("n_ctas", [8, 9, 16, 17, 152])
def test_merge_tree_fan_in(n_ctas):
    """One long request split over every CTA: 8 splits merge in one level,
    9 and more go through the two-level tree."""
    w = W.make_custom([6000], num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16, seed=n_ctas)
    _check(w, n_ctas=n_ctas)
    w2 = W.make_custom([3000, 5], q_tokens=4, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                       page_size=16, seed=n_ctas)
    _check(w2, n_ctas=n_ctas)
