"""Absorbed-MLA decode attention (tcgen05 / 2-CTA cluster path) on the GPU
against the fp64 oracle, through the C ABI."""
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


def _check(w, **kw):
    out, lse, err, _ = Dev(w).run(**kw)
    assert err == 0
    d_out, d_lse = compare(w, out, lse)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
    return out, lse


@pytest.mark.parametrize("n_workers", [1, 2, 5, None])
def test_mla_ragged_lengths(n_workers):
    _check(_mla([1, 63, 64, 65, 200, 0, 1000, 3000], seed=1), n_ctas=n_workers)


@pytest.mark.parametrize("n_workers", [5, None])
def test_mla_two_kernel_comparator(n_workers):
    # fixed splits written by every worker, merged by the separate combine kernel
    _check(_mla([1, 63, 64, 65, 200, 0, 1000, 3000], seed=1), n_ctas=n_workers, mode="fixed_split",
           two_kernel=True)


def _ramp_scores(w, step):
    """Scores rise by `step` (natural-log units) per 64-token block: q's rope
    columns are all 1 and key t's rope columns all 24 * step * (t // 64) / 64,
    so q.k / 24 gains step * (t // 64); the value columns are untouched."""
    q = W.bf16_bits_to_fp32(w.q)
    q[..., 512:] = 1.0
    w.q[...] = W.fp32_to_bf16_bits(q)
    P = w.page_size
    for b, L in enumerate(w.seqlens):
        for t0 in range(0, int(L), 64):
            pg = w.page_table[b, t0 // P]
            n = min(64, int(L) - t0)
            val = np.float32(24.0 * step * (t0 // 64) / 64.0)
            w.k_pages[pg, t0 % P:t0 % P + n, 0, 512:] = W.fp32_to_bf16_bits(np.full((n, 64), val, np.float32))


@pytest.mark.parametrize("n_workers", [1, 2, None])
def test_mla_rising_scores_move_the_reference(n_workers):
    # about 5.8 log2 units per block against the lazy threshold of 8: the
    # reference moves every block or two and the value CTA rescales O, across
    # single-block, odd-length and split segments
    w = _mla([3000, 64, 700, 1, 130, 2000], seed=6)
    _ramp_scores(w, 4.0)
    _check(w, n_ctas=n_workers)


def test_mla_many_one_block_requests():
    # every segment is a single block: Q is loaded for every block
    _check(_mla([1 + (7 * i) % 64 for i in range(41)], seed=7), n_ctas=3)


def test_mla_single_long_request_many_splits():
    _check(_mla([20000], seed=2))


def test_mla_page_size_128_and_shuffled_pages():
    _check(_mla([700, 129, 4096], seed=3, page_size=128, spare_pages=5))


def test_mla_constant_values_and_length_one():
    w = _mla([1, 300, 77], seed=4)
    w.k_pages[..., :512] = W.fp32_to_bf16_bits(np.full(w.k_pages[..., :512].shape, 0.75, np.float32))
    out, lse, err, _ = Dev(w).run()
    assert err == 0
    assert np.all(out.float().cpu().numpy() == 0.75)
    ro, rl = A.decode_workload(w)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL


def test_mla_repeatable_bits():
    w = _mla([5000, 333, 64], seed=5)
    d = Dev(w)
    o1, l1, _, ws = d.run()
    o2, l2, _, _ = d.run(ws=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
def test_mla_named_workload_full_size():
    """B=64, 128 heads, latent 576 / value 512, L ~ U[1024, 16384], P=64; rows
    sampled across every request (the oracle computes them one by one)."""
    w = W.make("mla_absorbed")
    out, lse, err, _ = Dev(w).run()
    assert err == 0
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([b * 128 + rng.choice(128, 6, replace=False) for b in range(w.batch)]))
    d_out, d_lse = compare(w, out, lse, rows=rows)
    assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
