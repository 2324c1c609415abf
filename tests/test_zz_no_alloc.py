"""The allocation-free entry point (skd_decode_attention_noalloc), for callers
that cannot allocate a workspace: its output must match the workspace entry
point's on the same inputs, on two calls in a row (the shared scratch array
keeps the previous call's contents, so the second call checks that the
counters and error word are cleared). Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import LSE_TOL, OUT_TOL, Dev

pytestmark = pytest.mark.gpu


def _max_diff(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(fin, np.isfinite(a))
    return float(np.abs(a[fin] - b[fin]).max()) if fin.any() else 0.0


def test_no_alloc_entry_matches_workspace_entry_on_two_calls():
    import sm_load_balancing_gb300 as skd
    from sm_load_balancing_gb300 import _native as N
    # ragged lengths, an empty request, items split across CTAs (merges)
    w = W.make_custom([1, 15, 700, 3000, 0, 129, 9000], num_q_heads=32, num_kv_heads=8,
                      head_dim_qk=128, page_size=16, seed=21)
    d = Dev(w)
    n = skd.sm_count()
    plan = skd.plan(w.seqlens, w.num_kv_heads, w.page_size, n).cuda()
    ref_out, ref_lse, err, _ = d.run(n_ctas=n, plan=plan)
    assert err == 0
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = N.lib().skd_decode_attention_noalloc(
            ctypes.byref(d.shape), d.q.data_ptr(), d.k.data_ptr(), d.v.data_ptr(), d.pt.data_ptr(),
            d.sl.data_ptr(), plan.data_ptr(), n, out.data_ptr(), lse.data_ptr(), stream.cuda_stream)
        assert st == N.SKD_OK
        torch.cuda.synchronize()
        assert _max_diff(out, ref_out) <= OUT_TOL
        assert _max_diff(lse, ref_lse) <= LSE_TOL


def test_no_alloc_entry_rejects_sizes_beyond_its_scratch():
    from sm_load_balancing_gb300 import _native as N
    lib = N.lib()
    # 8 kv heads x 16 rows x 131 floats per split, 2 splits per CTA: 2000 CTAs need ~134 MB
    s = N.Shape(batch=4, q_tokens=4, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                head_dim_v=128, page_size=16, max_pages_per_req=8, num_pages=32, v_row_stride=128,
                scale=0.088, causal=1, kind=0)
    assert lib.skd_workspace_bytes(ctypes.byref(s), 2000) > (32 << 20)
    fake = 1 << 20  # never dereferenced: the size check comes first
    st = lib.skd_decode_attention_noalloc(ctypes.byref(s), fake, fake, fake, fake, fake, fake, 2000,
                                          fake, fake, None)
    assert st == N.SKD_ESIZE
