"""Shared-prefix decode (prefix pass + suffix pass + state merge, all in the
library's kernels) on the GPU against the fp64 oracle of the full sequences."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev, compare

pytestmark = pytest.mark.gpu


def _run(w, n_ctas=None):
    import sm_load_balancing_gb300 as skd
    from sm_load_balancing_gb300.prefix import SharedPrefixDecode
    d = Dev(w)
    sp = SharedPrefixDecode(d.q, d.k, d.v, w.page_table, w.seqlens, w.prefix_groups, w.prefix_lens,
                            scale=w.scale, causal=w.causal, n_ctas=n_ctas)
    out, lse = sp(d.q)
    torch.cuda.synchronize()
    errs = [skd.read_error(x) for x in sp.workspaces()]
    return out, lse, errs, sp


@pytest.mark.parametrize("n_ctas", [3, None])
def test_groups_of_several_sizes_match_full_attention(n_ctas):
    # (one launch: virtual prefix requests and padded suffix requests in one batch)
    rng = np.random.default_rng(0)
    L = list(1024 + rng.integers(1, 600, size=12))
    w = W.make_custom(L, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16, seed=3)
    # a group of 5 (two stacked virtual requests), a group of 2, a group of 1, ungrouped requests
    w = W.share_prefix(w, [[0, 3, 4, 7, 9], [1, 2], [11]], [1024, 512, 1008])
    out, lse, errs, sp = _run(w, n_ctas)
    assert not any(errs) and sp.fused
    assert sp.V == 4
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)


def test_speculative_causal_rows():
    # T = 4 new tokens, causal among them; G = 4 -> one request per virtual request
    L = [700, 900, 640, 1000]
    w = W.make_custom(L, q_tokens=4, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16, seed=4)
    w = W.share_prefix(w, [[0, 1, 2, 3]], [512])
    out, lse, errs, sp = _run(w)
    assert not any(errs) and sp.R == 1 and not sp.fused  # causal: two launches
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)


def test_head_dim_64_and_all_requests_grouped():
    L = [300, 320, 290, 500, 333, 350, 301, 299]
    w = W.make_custom(L, num_q_heads=16, num_kv_heads=2, head_dim_qk=64, page_size=32, seed=5)
    w = W.share_prefix(w, [[0, 1, 2, 3, 4, 5, 6, 7]], [256])  # G = 8 -> 2 requests per virtual request
    out, lse, errs, sp = _run(w)
    assert not any(errs) and sp.V == 4
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)


def test_one_and_two_launch_paths_agree():
    from sm_load_balancing_gb300.prefix import SharedPrefixDecode
    L = [900, 1100, 700, 1300]
    w = W.make_custom(L, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16, seed=8)
    w = W.share_prefix(w, [[0, 1, 2]], [640])
    d = Dev(w)
    res = []
    for fuse in (True, False):
        sp = SharedPrefixDecode(d.q, d.k, d.v, w.page_table, w.seqlens, w.prefix_groups, w.prefix_lens,
                                scale=w.scale, causal=False, fuse=fuse)
        assert sp.fused == fuse and sp.launches() == (3 if fuse else 4)
        o, l = sp(d.q)
        torch.cuda.synchronize()
        d_out, d_lse = compare(w, o, l)
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (fuse, d_out, d_lse)
        res.append((o.float(), l))
    assert (res[0][0] - res[1][0]).abs().max().item() <= OUT_TOL


def test_merge_with_no_groups_is_the_plain_decode():
    w = W.make_custom([100, 2000, 37], num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16, seed=6)
    w = W.dataclasses.replace(w, prefix_groups=[], prefix_lens=[])
    out, lse, errs, sp = _run(w)
    assert sp.V == 0 and errs == [0] and not sp.fused
    d = Dev(w)
    o2, l2, err, _ = d.run()
    assert err == 0 and torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.slow
def test_named_shared_prefix_workload():
    w = W.make("shared_prefix_gqa")
    out, lse, errs, sp = _run(w)
    assert not any(errs)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([b * 32 + rng.choice(32, 4, replace=False) for b in range(w.batch)]))
    d_out, d_lse = compare(w, out, lse, rows=rows)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
