"""The device planner and the attention launch captured together in one CUDA
graph ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 7: a graph
replays fixed launches with fixed buffers). The request lengths live in a
device buffer that the caller rewrites between replays; the graph recomputes
the plan on the device each time, so a replay after new lengths must match the
oracle for those lengths. Run with and without programmatic dependent launch."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev, compare

pytestmark = pytest.mark.gpu

CASES = {
    "gqa": dict(seqlens=[700, 33, 4100, 129, 2048], num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                page_size=16),
    "gqa_causal": dict(seqlens=[300, 2500, 77], q_tokens=4, num_q_heads=32, num_kv_heads=8,
                       head_dim_qk=128, page_size=16),
    "mla": dict(seqlens=[1000, 64, 3000, 1, 700], num_q_heads=128, num_kv_heads=1, head_dim_qk=576,
                head_dim_v=512, page_size=64, mla=True),
}
# second replay: every request shorter (the page table still covers the first lengths)
SHORTER = {"gqa": [699, 16, 1, 128, 2000], "gqa_causal": [4, 1999, 77], "mla": [999, 63, 2, 1, 640]}


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("case", sorted(CASES))
def test_graph_replays_plan_and_attention(case, pdl):
    import sm_load_balancing_gb300 as skd
    skd.set_pdl(pdl)
    try:
        w = W.make_custom(seed=11, **CASES[case])
        d = Dev(w)
        n = skd.default_ctas(d.shape)
        c, al = skd.default_seg_cost(d.shape), skd.default_align(d.shape)
        hkv = d.shape.num_kv_heads
        plan = skd.plan_device(d.sl, hkv, w.page_size, n, seg_cost=c, align=al)
        ws = skd.workspace(d.shape, n)
        kw = dict(scale=w.scale, causal=w.causal, n_ctas=n, shape=d.shape)
        out, lse = skd.decode_attention(d.q, d.k, d.v, d.pt, d.sl, plan, ws, **kw)  # eager, sets attributes
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            skd.plan_device(d.sl, hkv, w.page_size, n, out=plan, seg_cost=c, align=al)
            skd.decode_attention(d.q, d.k, d.v, d.pt, d.sl, plan, ws, out=out, lse=lse, **kw)
        torch.cuda.current_stream().wait_stream(s)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert skd.read_error(ws) == 0
        d_out, d_lse = compare(w, out, lse)
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
        # new lengths in place, same graph
        d.sl.copy_(torch.tensor(SHORTER[case], dtype=torch.int32))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert skd.read_error(ws) == 0
        w2 = dataclasses.replace(w, seqlens=np.array(SHORTER[case], dtype=np.int32))
        d_out, d_lse = compare(w2, out, lse)
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (d_out, d_lse)
    finally:
        skd.set_pdl(True)
