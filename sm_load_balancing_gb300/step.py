"""One decode step captured as a CUDA graph, for a serving loop with fixed
batch slots.

The graph holds, in order: the copies of the step's inputs from pinned host
buffers (queries, page table, request lengths, and for the sparse form the
top-k lists), the device planner over the new lengths, the decode launch, and
the copies of out / lse back into pinned host buffers. The caller writes the
next step's inputs into the ``*_host`` tensors and calls ``run()``: one graph
replay instead of a host plan and eight separately issued operations. The
KV cache stays resident on the device; only its contents change between
steps.

"GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 7: a CUDA graph
replays a fixed sequence of launches and copies on fixed buffers, which takes
the per-launch host cost off the step. Every step of the attention itself
runs in the library's kernels; this module only allocates buffers and
records the sequence.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch


class DecodeStep:
    """A captured decode step over ``batch`` request slots.

    ``q_like``: a bf16 tensor of the step's query shape [B, T, Hq, Dk]
    (values unused); ``k_pages`` / ``v_pages``: the resident paged cache
    (``v_pages`` None for absorbed MLA); ``max_pages``: page-table width.
    ``topk``: for the sparse (top-k) MLA form, the list capacity K per request.
    Plan settings default to the library's per-kind defaults.
    """

    def __init__(self, q_like: torch.Tensor, k_pages: torch.Tensor, v_pages: Optional[torch.Tensor],
                 max_pages: int, *, scale: float, causal: Optional[bool] = None, topk: Optional[int] = None,
                 n_ctas: Optional[int] = None, seg_cost: Optional[int] = None, align: Optional[int] = None):
        from . import (decode_attention, decode_attention_sparse, default_align, default_ctas, default_seg_cost,
                       make_shape, plan_bytes, plan_device, workspace)
        if q_like.dim() != 4 or q_like.dtype != torch.bfloat16:
            raise ValueError("q_like must be a bf16 tensor [B, T, Hq, Dk]")
        if k_pages.device.type != "cuda" or k_pages.dtype != torch.bfloat16:
            raise ValueError("k_pages must be a CUDA bf16 tensor (the resident cache)")
        if v_pages is not None and (v_pages.device != k_pages.device or v_pages.dtype != torch.bfloat16):
            raise ValueError("v_pages must be a bf16 tensor on k_pages' device")
        if int(max_pages) < 1:
            raise ValueError("max_pages must be at least 1")
        dev = k_pages.device
        B, T, Hq = int(q_like.shape[0]), int(q_like.shape[1]), int(q_like.shape[2])
        if causal is None:
            causal = T > 1
        self.sparse = topk is not None
        if self.sparse and (v_pages is not None or causal or int(topk) < 1):
            raise ValueError("the sparse form is absorbed MLA without a causal mask (v_pages None, topk >= 1)")
        pin = dict(pin_memory=True)
        # pinned host inputs and outputs (the caller's side of the step)
        self.q_host = torch.zeros(tuple(q_like.shape), dtype=torch.bfloat16, **pin)
        self.page_table_host = torch.zeros(B, int(max_pages), dtype=torch.int32, **pin)
        self.seqlens_host = torch.zeros(B, dtype=torch.int32, **pin)
        if self.sparse:
            self.topk_idx_host = torch.zeros(B, int(topk), dtype=torch.int32, **pin)
            self.topk_len_host = torch.zeros(B, dtype=torch.int32, **pin)
        # device copies
        self.q = torch.zeros_like(self.q_host, device=dev)
        self.page_table = torch.zeros_like(self.page_table_host, device=dev)
        self.seqlens = torch.zeros_like(self.seqlens_host, device=dev)
        if self.sparse:
            self.topk_idx = torch.zeros_like(self.topk_idx_host, device=dev)
            self.topk_len = torch.zeros_like(self.topk_len_host, device=dev)
        self.shape = make_shape(self.q, k_pages, v_pages, self.page_table, scale=scale, causal=causal)
        self.n = default_ctas(self.shape) if n_ctas is None else int(n_ctas)
        self.seg_cost = default_seg_cost(self.shape, sparse=self.sparse) if seg_cost is None else int(seg_cost)
        self.align = default_align(self.shape) if align is None else int(align)
        hkv = self.shape.num_kv_heads
        P = int(k_pages.shape[1])
        self.plan = torch.zeros(plan_bytes(B, hkv, self.n) // 4, dtype=torch.int32, device=dev)
        self.ws = workspace(self.shape, self.n, dev)
        self.out = torch.zeros(B, T, Hq, self.shape.head_dim_v, dtype=torch.bfloat16, device=dev)
        self.lse = torch.zeros(B, T, Hq, dtype=torch.float32, device=dev)
        self.out_host = torch.zeros(tuple(self.out.shape), dtype=torch.bfloat16, **pin)
        self.lse_host = torch.zeros(tuple(self.lse.shape), dtype=torch.float32, **pin)
        lens = self.topk_len if self.sparse else self.seqlens

        def record():
            self.q.copy_(self.q_host, non_blocking=True)
            self.page_table.copy_(self.page_table_host, non_blocking=True)
            self.seqlens.copy_(self.seqlens_host, non_blocking=True)
            if self.sparse:
                self.topk_idx.copy_(self.topk_idx_host, non_blocking=True)
                self.topk_len.copy_(self.topk_len_host, non_blocking=True)
            plan_device(lens, hkv, P, self.n, out=self.plan, seg_cost=self.seg_cost, align=self.align)
            if self.sparse:
                decode_attention_sparse(self.q, k_pages, self.page_table, self.seqlens, self.topk_idx,
                                        self.topk_len, self.plan, self.ws, scale=scale, n_ctas=self.n,
                                        out=self.out, lse=self.lse, shape=self.shape)
            else:
                decode_attention(self.q, k_pages, v_pages, self.page_table, self.seqlens, self.plan, self.ws,
                                 scale=scale, causal=causal, n_ctas=self.n, out=self.out, lse=self.lse,
                                 shape=self.shape)
            self.out_host.copy_(self.out, non_blocking=True)
            self.lse_host.copy_(self.lse, non_blocking=True)

        # one eager pass (all-empty requests) sets the kernels' attributes, then capture
        self.stream = torch.cuda.Stream(device=dev)
        self.stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(self.stream):
            record()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            record()

    def host_to_device_bytes(self) -> int:
        """Bytes the step copies to the device."""
        t = [self.q_host, self.page_table_host, self.seqlens_host]
        if self.sparse:
            t += [self.topk_idx_host, self.topk_len_host]
        return sum(x.numel() * x.element_size() for x in t)

    def device_to_host_bytes(self) -> int:
        return self.out_host.numel() * 2 + self.lse_host.numel() * 4

    def run(self, sync: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
        """Replay the step on its own stream, after the work already queued on
        the caller's current stream (e.g. writes into the KV cache); with
        ``sync``, wait for it. Returns the pinned host (out, lse). Without
        ``sync`` the host buffers must not be touched until the step's stream
        has finished."""
        self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        with torch.cuda.stream(self.stream):  # a replay runs on the current stream
            self.graph.replay()
        if sync:
            self.stream.synchronize()
        return self.out_host, self.lse_host

    def error(self) -> int:
        """The device error word of the step's workspace (0: no error)."""
        from . import read_error
        return read_error(self.ws)
