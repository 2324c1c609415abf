"""Shared-prefix decode composed from the library's kernels.

Requests that share a prefix (the same first pages of KV cache) read it once
("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", results: shared-prefix
decode, Fig. 11): the query rows of up to ``16 // (G * T)`` requests of a group
are stacked as the tokens of one virtual request that attends (without causal
mask) to the prefix only; every request also attends to its own suffix; a
merge kernel combines the two (out, lse) states row by row. Without a causal
mask (T = 1) the virtual requests and the suffix requests (their query rows
padded to the same token count, which the 16-row MMA tile pads anyway) form one
batch with one Stream-K plan, so both kinds of work share one launch; with a
causal mask they are two launches. All attention and merge arithmetic runs in
the CUDA kernels (decode, ``skd_gather_rows``, ``skd_merge_states``); this
module only builds index arrays on the host.

Requirements: each group's prefix length is a positive multiple of the page
size, the members' page tables list the same pages for it, and every member
has at least ``q_tokens`` tokens after it (the new tokens are in the suffix).
GQA layout only (the decode kernel holds at most 16 query rows per kv head).
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import _native as N


@dataclasses.dataclass
class PrefixLayout:
    rows_per_virtual: int          # members stacked into one virtual request
    virtual: List[tuple]           # (group index, member request ids)
    q_rows: np.ndarray             # int32 [V * R * T]: source row b*T + t of each stacked row, or -1
    v_seqlens: np.ndarray          # int32 [V]: the prefix length of the group
    v_page_table: np.ndarray       # int32 [V][max_pages]: the prefix pages
    s_seqlens: np.ndarray          # int32 [B]: tokens after the request's prefix
    s_page_table: np.ndarray       # int32 [B][max_pages]: the pages after it
    a_rows: np.ndarray             # int32 [B * T * Hq]: row of the prefix result, or -1


def shared_prefix_layout(seqlens, page_table, groups: Sequence[Sequence[int]], prefix_lens: Sequence[int],
                         page_size: int, q_tokens: int, num_q_heads: int, num_kv_heads: int) -> PrefixLayout:
    """Index arrays for ``SharedPrefixDecode`` (host only, no attention math)."""
    sl = np.asarray(seqlens, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int32)
    B, mp = pt.shape
    T, Hq = int(q_tokens), int(num_q_heads)
    G = Hq // int(num_kv_heads)
    R = max(1, 16 // (G * T))
    if len(groups) != len(prefix_lens):
        raise ValueError("one prefix length per group")
    seen = set()
    plen = np.zeros(B, dtype=np.int64)
    for gi, (mem, lp) in enumerate(zip(groups, prefix_lens)):
        lp = int(lp)
        if lp <= 0 or lp % page_size:
            raise ValueError(f"group {gi}: prefix length {lp} is not a positive multiple of {page_size}")
        npg = lp // page_size
        for b in mem:
            if b in seen or not 0 <= b < B:
                raise ValueError(f"group {gi}: request {b} repeated or out of range")
            seen.add(b)
            if sl[b] - lp < T:
                raise ValueError(f"request {b}: fewer than {T} tokens after its prefix")
            if not np.array_equal(pt[b, :npg], pt[mem[0], :npg]):
                raise ValueError(f"group {gi}: request {b} does not share the prefix pages")
            plen[b] = lp
    virtual = []
    for gi, mem in enumerate(groups):
        mem = list(mem)
        for c in range(0, len(mem), R):
            virtual.append((gi, mem[c:c + R]))
    V = len(virtual)
    q_rows = np.full(max(V * R * T, 1), -1, dtype=np.int32)[:V * R * T]
    v_sl = np.zeros(V, dtype=np.int32)
    v_pt = np.full((max(V, 1), mp), -1, dtype=np.int32)[:V]
    a_rows = np.full(B * T * Hq, -1, dtype=np.int32)
    h = np.arange(Hq)
    for v, (gi, mem) in enumerate(virtual):
        lp = int(prefix_lens[gi])
        v_sl[v] = lp
        v_pt[v, :lp // page_size] = pt[mem[0], :lp // page_size]
        for m, b in enumerate(mem):
            for t in range(T):
                q_rows[(v * R + m) * T + t] = b * T + t
                a_rows[(b * T + t) * Hq + h] = ((v * R + m) * T + t) * Hq + h
    s_sl = (sl - plen).astype(np.int32)
    s_pt = np.full_like(pt, -1)
    for b in range(B):
        off = int(plen[b]) // page_size
        s_pt[b, :mp - off] = pt[b, off:]
    return PrefixLayout(R, virtual, q_rows, v_sl, v_pt, s_sl, s_pt, a_rows)


class SharedPrefixDecode:
    """Prepared shared-prefix decode for fixed lengths and groups; call with
    the batch's queries to run prefix pass, suffix pass and merge (``fuse``:
    one decode launch for both when there is no causal mask).

    q: bf16 [B][T][Hq][D]; k_pages / v_pages: the paged cache (GQA);
    page_table / seqlens: host int32 arrays of the whole requests."""

    def __init__(self, q_like, k_pages, v_pages, page_table, seqlens, groups, prefix_lens, *, scale: float,
                 causal: Optional[bool] = None, n_ctas: Optional[int] = None, fuse: bool = True):
        from . import default_ctas, make_shape, plan, workspace
        B, T, Hq, D = (int(x) for x in q_like.shape)
        dev = q_like.device
        Hkv = int(k_pages.shape[2])
        P = int(k_pages.shape[1])
        if causal is None:
            causal = T > 1
        lay = shared_prefix_layout(seqlens, page_table, groups, prefix_lens, P, T, Hq, Hkv)
        self.layout = lay
        self.k, self.v, self.scale, self.causal = k_pages, v_pages, float(scale), bool(causal)
        R, V = lay.rows_per_virtual, len(lay.virtual)
        self.V, self.R, self.T, self.Hq, self.D, self.B = V, R, T, Hq, D, B
        self.fused = fuse and (not causal) and V > 0
        if self.fused:
            # one batch: V virtual prefix requests, then the B suffix requests
            # with their T query rows padded to R*T tokens
            TT = R * T
            qr = np.full((V + B) * TT, -1, dtype=np.int32)
            qr[:V * TT] = lay.q_rows
            b_rows = np.zeros(B * T * Hq, dtype=np.int32)
            h = np.arange(Hq)
            for b in range(B):
                for t in range(T):
                    qr[(V + b) * TT + t] = b * T + t
                    b_rows[(b * T + t) * Hq + h] = ((V + b) * TT + t) * Hq + h
            self.c_rows = torch.from_numpy(qr).to(dev)
            self.b_rows = torch.from_numpy(b_rows).to(dev)
            c_pt = np.ascontiguousarray(np.concatenate([lay.v_page_table, lay.s_page_table]))
            c_sl = np.concatenate([lay.v_seqlens, lay.s_seqlens]).astype(np.int32)
            self.c_pt = torch.from_numpy(c_pt).to(dev)
            self.c_sl = torch.from_numpy(c_sl).to(dev)
            self.qc = torch.empty(V + B, TT, Hq, D, dtype=torch.bfloat16, device=dev)
            self.shape_c = make_shape(self.qc, k_pages, v_pages, self.c_pt, scale=scale, causal=False)
            n = default_ctas(self.shape_c) if n_ctas is None else int(n_ctas)
            self.n = n
            self.plan_c = plan(c_sl, Hkv, P, n).to(dev)
            self.ws_c = workspace(self.shape_c, n)
            self.out_c = torch.empty(V + B, TT, Hq, D, dtype=torch.bfloat16, device=dev)
            self.lse_c = torch.empty(V + B, TT, Hq, dtype=torch.float32, device=dev)
            self.a_rows = torch.from_numpy(lay.a_rows).to(dev)
            return
        self.q_rows = torch.from_numpy(lay.q_rows).to(dev)
        self.v_pt = torch.from_numpy(np.ascontiguousarray(lay.v_page_table)).to(dev)
        self.v_sl = torch.from_numpy(lay.v_seqlens).to(dev)
        self.s_pt = torch.from_numpy(lay.s_page_table).to(dev)
        self.s_sl = torch.from_numpy(lay.s_seqlens).to(dev)
        self.a_rows = torch.from_numpy(lay.a_rows).to(dev)
        self.qv = torch.empty(max(V, 1), R * T, Hq, D, dtype=torch.bfloat16, device=dev)[:V]
        self.shape_s = make_shape(q_like, k_pages, v_pages, self.s_pt, scale=scale, causal=causal)
        n = default_ctas(self.shape_s) if n_ctas is None else int(n_ctas)
        self.n = n
        self.plan_s = plan(lay.s_seqlens, Hkv, P, n).to(dev)
        self.ws_s = workspace(self.shape_s, n)
        self.out_s = torch.empty(B, T, Hq, D, dtype=torch.bfloat16, device=dev)
        self.lse_s = torch.empty(B, T, Hq, dtype=torch.float32, device=dev)
        if V:
            self.shape_v = make_shape(self.qv, k_pages, v_pages, self.v_pt, scale=scale, causal=False)
            self.plan_v = plan(lay.v_seqlens, Hkv, P, n).to(dev)
            self.ws_v = workspace(self.shape_v, n)
            self.out_v = torch.empty(V, R * T, Hq, D, dtype=torch.bfloat16, device=dev)
            self.lse_v = torch.empty(V, R * T, Hq, dtype=torch.float32, device=dev)

    def launches(self) -> int:
        """Kernels of ours per call: gather + decode + merge (fused), else the
        suffix decode, with a prefix pass its gather + decode, then the merge."""
        return 3 if self.fused else (4 if self.V else 2)

    def workspaces(self):
        """The decode workspaces of this composition (for reading error words)."""
        if self.fused:
            return [self.ws_c]
        return [self.ws_s] + ([self.ws_v] if self.V else [])

    def kv_tokens(self) -> int:
        """KV rows read per call: each virtual request's prefix once, every suffix once."""
        return int(self.layout.v_seqlens.astype(np.int64).sum() + self.layout.s_seqlens.astype(np.int64).sum())

    def __call__(self, q, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None):
        from . import _stream_ptr, decode_attention
        lib = N.lib()
        st = _stream_ptr(stream)
        if out is None:
            out = torch.empty(self.B, self.T, self.Hq, self.D, dtype=torch.bfloat16, device=q.device)
        if lse is None:
            lse = torch.empty(self.B, self.T, self.Hq, dtype=torch.float32, device=q.device)
        if self.fused:
            N.check("skd_gather_rows", lib.skd_gather_rows(
                self.qc.data_ptr(), q.data_ptr(), self.c_rows.data_ptr(), self.qc.shape[0] * self.qc.shape[1],
                self.Hq * self.D * 2, st))
            decode_attention(self.qc, self.k, self.v, self.c_pt, self.c_sl, self.plan_c, self.ws_c,
                             scale=self.scale, causal=False, n_ctas=self.n, out=self.out_c, lse=self.lse_c,
                             shape=self.shape_c, stream=stream)
            N.check("skd_merge_states", lib.skd_merge_states(
                self.out_c.data_ptr(), self.lse_c.data_ptr(), self.a_rows.data_ptr(), self.out_c.data_ptr(),
                self.lse_c.data_ptr(), self.b_rows.data_ptr(), out.data_ptr(), lse.data_ptr(),
                self.B * self.T * self.Hq, self.D, st))
            return out, lse
        decode_attention(q, self.k, self.v, self.s_pt, self.s_sl, self.plan_s, self.ws_s, scale=self.scale,
                         causal=self.causal, n_ctas=self.n, out=self.out_s, lse=self.lse_s, shape=self.shape_s,
                         stream=stream)
        if self.V:
            N.check("skd_gather_rows", lib.skd_gather_rows(
                self.qv.data_ptr(), q.data_ptr(), self.q_rows.data_ptr(), self.V * self.R * self.T,
                self.Hq * self.D * 2, st))
            decode_attention(self.qv, self.k, self.v, self.v_pt, self.v_sl, self.plan_v, self.ws_v,
                             scale=self.scale, causal=False, n_ctas=self.n, out=self.out_v, lse=self.lse_v,
                             shape=self.shape_v, stream=stream)
            a_out, a_lse, a_rows = self.out_v.data_ptr(), self.lse_v.data_ptr(), self.a_rows.data_ptr()
        else:
            a_out, a_lse, a_rows = self.out_s.data_ptr(), self.lse_s.data_ptr(), self.a_rows.data_ptr()
        N.check("skd_merge_states", lib.skd_merge_states(
            a_out, a_lse, a_rows, self.out_s.data_ptr(), self.lse_s.data_ptr(), None, out.data_ptr(),
            lse.data_ptr(), self.B * self.T * self.Hq, self.D, st))
        return out, lse
