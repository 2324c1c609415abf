"""Helpers for the GPU tests: move a seeded workload to the device, run the
library through its C ABI, and compare with the fp64 oracle."""
import numpy as np
import torch

import workloads as W
from oracle import attention as A

OUT_TOL = 1e-2   # max-abs on bf16 outputs
LSE_TOL = 1e-3   # max-abs on fp32 lse


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class Dev:
    """A workload resident on cuda:0."""

    def __init__(self, w):
        import sm_load_balancing_gb300 as skd
        self.skd = skd
        self.w = w
        self.q = bf16(w.q).cuda()
        self.k = bf16(w.k_pages).cuda()
        self.v = None if w.mla else bf16(w.v_pages).cuda()
        self.pt = torch.from_numpy(w.page_table).cuda()
        self.sl = torch.from_numpy(w.seqlens).cuda()
        self.shape = skd.make_shape(self.q, self.k, self.v, self.pt, scale=w.scale, causal=w.causal)

    def run(self, n_ctas=None, mode="streamk", plan=None, ws=None, out=None, lse=None, seg_cost=None,
            two_kernel=False, align=None):
        skd = self.skd
        n = skd.default_ctas(self.shape) if n_ctas is None else n_ctas
        if plan is None:
            if seg_cost is None:
                seg_cost = skd.default_seg_cost(self.shape) if mode == "streamk" else 0
            if align is None:
                align = skd.default_align(self.shape) if mode == "streamk" else 1
            plan = skd.plan(self.w.seqlens, self.shape.num_kv_heads, self.w.page_size, n, mode,
                            seg_cost=seg_cost, align=align).cuda()
        if ws is None:
            ws = skd.workspace(self.shape, n)
        o, l = skd.decode_attention(self.q, self.k, self.v, self.pt, self.sl, plan, ws,
                                    scale=self.w.scale, causal=self.w.causal, n_ctas=n,
                                    shape=self.shape, out=out, lse=lse, two_kernel=two_kernel)
        torch.cuda.synchronize()
        err = skd.read_error(ws)
        return o, l, err, ws


def to_np(out, lse):
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(w, out, lse, rows=None, ref=None):
    """Max-abs errors vs the oracle (all rows, or the flattened row ids given)."""
    o, l = to_np(out, lse)
    if ref is None:
        ref = A.decode_workload(w, rows=rows)
    ro, rl = ref
    if rows is not None:
        o = o.reshape(-1, w.head_dim_v)[rows]
        l = l.reshape(-1)[rows]
    ro = ro.reshape(o.shape)
    rl = rl.reshape(l.shape)
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(l)), "lse finiteness differs"
    # Where |out| >= 2 one bf16 ulp (>= 2^-6) is coarser than the 1e-2 bound
    # itself, so there the bound is one ulp of the reference value; such values
    # only arise in rows that see a handful of keys.
    big = np.abs(ro) >= 2.0
    if big.any():
        ulp = np.exp2(np.floor(np.log2(np.abs(ro[big]))) - 7)
        assert np.all(np.abs(o[big] - ro[big]) <= ulp), "more than one bf16 ulp off"
    d_out = float(np.abs(o - ro)[~big].max()) if (~big).any() else 0.0
    d_lse = float(np.abs(l[fin] - rl[fin]).max()) if fin.any() else 0.0
    assert np.all(l[~fin] == -np.inf)
    return d_out, d_lse
