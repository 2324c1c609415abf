"""Sparse (top-k) absorbed-MLA decode on the GPU against the fp64 sparse
oracle, through the C ABI (skd_decode_attention_sparse)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev, compare

pytestmark = pytest.mark.gpu


def _mla(seqlens, seed=0, **kw):
    return W.make_custom(seqlens, mla=True, num_q_heads=128, head_dim_qk=576, head_dim_v=512,
                         page_size=kw.pop("page_size", 64), scale=1.0 / 24.0, seed=seed, **kw)


def _run(w, n_ctas=None, d=None):
    import sm_load_balancing_gb300 as skd
    d = d or Dev(w)
    ti = torch.from_numpy(w.topk_idx).cuda()
    tl = torch.from_numpy(w.topk_len).cuda()
    n = skd.default_ctas(d.shape) if n_ctas is None else n_ctas
    plan = skd.plan(w.topk_len, 1, w.page_size, n, seg_cost=skd.default_seg_cost(d.shape, sparse=True),
                    align=skd.default_align(d.shape)).cuda()
    ws = skd.workspace(d.shape, n)
    out, lse = skd.decode_attention_sparse(d.q, d.k, d.pt, d.sl, ti, tl, plan, ws, scale=w.scale, n_ctas=n,
                                           shape=d.shape)
    torch.cuda.synchronize()
    return out, lse, skd.read_error(ws)


def _check(w, **kw):
    out, lse, err = _run(w, **kw)
    assert err == 0
    d_out, d_lse = compare(w, out, lse, ref=A.decode_sparse_workload(w))
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
    return out, lse


@pytest.mark.parametrize("n_workers", [1, 3, None])
@pytest.mark.parametrize("k", [1, 100, 2048])
def test_sparse_ragged(k, n_workers):
    # requests shorter than k list every position; one request lists nothing
    w = W.select_topk(_mla([3000, 65, 0, 700, 1, 2600], seed=k), k)
    _check(w, n_ctas=n_workers)


def test_sparse_page_size_128_shuffled_pages():
    w = W.select_topk(_mla([5000, 129, 4096], seed=3, page_size=128, spare_pages=5), 777)
    _check(w)


def test_sparse_repeats_and_short_lists():
    w = _mla([400, 90], seed=4)
    idx = np.zeros((2, 130), np.int32)
    idx[0, :130] = np.concatenate([np.arange(0, 400, 4), np.full(30, 17)])  # position 17 listed 31 times
    idx[1, :5] = [89, 0, 45, 45, 3]
    w = W.dataclasses.replace(w, topk_idx=idx, topk_len=np.array([130, 5], np.int32))
    _check(w, n_ctas=2)


def test_listing_every_position_matches_dense_bits():
    # the same keys in the same order, through the gather instead of TMA
    w = _mla([1000, 64, 3000, 7], seed=5)
    idx = np.zeros((w.batch, 3000), np.int32)
    for b, L in enumerate(w.seqlens):
        idx[b, :L] = np.arange(L)
    ws_ = W.dataclasses.replace(w, topk_idx=idx, topk_len=w.seqlens.copy())
    d = Dev(ws_)
    so, sl, err = _run(ws_, d=d)
    assert err == 0
    import sm_load_balancing_gb300 as skd
    do, dl, err2, _ = d.run(seg_cost=skd.default_seg_cost(d.shape, sparse=True))  # the same plan
    assert err2 == 0
    assert torch.equal(so, do) and torch.equal(sl, dl)


def test_out_of_range_position_is_reported():
    import sm_load_balancing_gb300 as skd
    w = W.select_topk(_mla([300, 200], seed=6), 50)
    idx = w.topk_idx.copy()
    idx[1, 7] = 200  # == seqlens[1]
    w = W.dataclasses.replace(w, topk_idx=idx)
    _, _, err = _run(w, n_ctas=2)
    assert err & skd.SKD_DEVERR_INDEX


def test_rising_scores_sparse():
    from tests.test_gpu_mla import _ramp_scores
    w = _mla([3000, 700, 2000], seed=7)
    _ramp_scores(w, 4.0)
    _check(W.select_topk(w, 1500), n_ctas=2)


@pytest.mark.slow
def test_sparse_named_workload_full_size():
    """B=64, 128 heads, latent 576 / value 512, L ~ U[1024, 16384], top-2048
    positions per request; rows sampled across every request."""
    w = W.make("mla_sparse_top2048")
    out, lse, err = _run(w)
    assert err == 0
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([b * 128 + rng.choice(128, 6, replace=False) for b in range(w.batch)]))
    d_out, d_lse = compare(w, out, lse, rows=rows, ref=A.decode_sparse_workload(w, rows=rows))
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
