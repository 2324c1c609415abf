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
