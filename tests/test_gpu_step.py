"""The captured decode step (sm_load_balancing_gb300.step.DecodeStep): pinned
host inputs -> device copies -> device planner -> decode -> pinned host
outputs, replayed as one CUDA graph. Each replay is checked against the fp64
oracle for the inputs written before it, and against an eager launch with the
host planner's plan (same plan bytes, so the same bits)."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev, bf16, compare

pytestmark = pytest.mark.gpu

CASES = {
    "gqa": dict(seqlens=[700, 33, 4100, 0, 2048], num_q_heads=32, num_kv_heads=8, head_dim_qk=128, page_size=16),
    "gqa_causal": dict(seqlens=[300, 2500, 77], q_tokens=4, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                       page_size=16),
    "mla": dict(seqlens=[1000, 64, 3000, 1, 700], num_q_heads=128, num_kv_heads=1, head_dim_qk=576,
                head_dim_v=512, page_size=64, mla=True),
}
SHORTER = {"gqa": [699, 16, 1, 0, 2000], "gqa_causal": [4, 1999, 77], "mla": [999, 63, 2, 1, 640]}


def _fill(step, w):
    step.q_host.copy_(bf16(w.q))
    step.page_table_host.copy_(torch.from_numpy(w.page_table))
    step.seqlens_host.copy_(torch.from_numpy(w.seqlens))
    if w.sparse:
        step.topk_idx_host.zero_()
        step.topk_idx_host[:, :w.topk_idx.shape[1]].copy_(torch.from_numpy(w.topk_idx))
        step.topk_len_host.copy_(torch.from_numpy(w.topk_len))


@pytest.mark.parametrize("case", sorted(CASES))
def test_step_replays_match_oracle_and_eager(case):
    from sm_load_balancing_gb300.step import DecodeStep
    w = W.make_custom(seed=21, **CASES[case])
    d = Dev(w)
    step = DecodeStep(d.q, d.k, d.v, w.page_table.shape[1], scale=w.scale, causal=w.causal)
    for ww in (w, dataclasses.replace(w, seqlens=np.array(SHORTER[case], dtype=np.int32),
                                      q=W.make_custom(seed=22, **CASES[case]).q)):
        _fill(step, ww)
        out_h, lse_h = step.run()
        # run() returns with the step complete: nothing left on either stream
        assert step.stream.query() and torch.cuda.current_stream().query()
        assert step.error() == 0
        d_out, d_lse = compare(ww, out_h, lse_h)
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
        # the eager path with the host planner's plan gives the same bits
        de = Dev(ww)
        eo, el, err, _ = de.run()
        assert err == 0
        assert torch.equal(eo.cpu(), out_h) and torch.equal(el.cpu(), lse_h)
    assert step.host_to_device_bytes() == (w.q.size * 2 + w.page_table.size * 4 + w.batch * 4)


def test_step_sparse_mla():
    from sm_load_balancing_gb300.step import DecodeStep
    base = W.make_custom([3000, 65, 0, 700, 2600], mla=True, num_q_heads=128, head_dim_qk=576, head_dim_v=512,
                         page_size=64, scale=1.0 / 24.0, seed=23)
    d = Dev(base)
    step = DecodeStep(d.q, d.k, None, base.page_table.shape[1], scale=base.scale, causal=False, topk=2048)
    for k in (2048, 100):
        w = W.select_topk(base, k, seed=k)
        _fill(step, w)
        out_h, lse_h = step.run()
        assert step.error() == 0
        d_out, d_lse = compare(w, out_h, lse_h, ref=A.decode_sparse_workload(w))
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
