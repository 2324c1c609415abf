"""Stream-K split-KV decode attention over a paged KV cache, for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libskdecode.so`` (``include/skdecode.h``).
Every step of the hot path runs in the library's CUDA kernels; this module only
checks dtypes/devices and passes raw pointers, sizes and the current stream.
PyTorch is used for device memory and streams.

    plan = skd.plan(seqlens_cpu, num_kv_heads, page_size)        # host planner
    plan_dev = plan.cuda()                                         # or skd.plan_device(...)
    ws = skd.workspace(q, k_pages, v_pages, n_ctas)                # zeroed once
    out, lse = skd.decode_attention(q, k_pages, v_pages, page_table, seqlens_dev,
                                    plan_dev, ws, scale=..., causal=...)
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _native as N
from ._native import (SKD_DEVERR_INDEX, SKD_DEVERR_PAGE, SKD_DEVERR_PLAN, SKD_DEVERR_SEQLEN,
                      SKD_DEVERR_TIMEOUT, SKD_GRANULE, SkdError)

__all__ = ["plan", "plan_device", "plan_bytes", "workspace", "decode_attention", "decode_attention_sparse",
           "read_error", "sm_count", "default_ctas", "default_seg_cost", "default_align", "make_shape", "set_pdl", "SkdError",
           "SKD_GRANULE", "SKD_DEVERR_PLAN", "SKD_DEVERR_SEQLEN", "SKD_DEVERR_PAGE", "SKD_DEVERR_TIMEOUT",
           "SKD_DEVERR_INDEX"]

_MODES = {"streamk": N.SKD_PLAN_STREAMK, "round_robin": N.SKD_PLAN_ROUND_ROBIN,
          "fixed_split": N.SKD_PLAN_FIXED_SPLIT}


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> Optional[int]:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream or None


def sm_count(device: Optional[int] = None) -> int:
    dev = torch.cuda.current_device() if device is None else int(device)
    v = ctypes.c_int(0)
    N.check("skd_device_sm_count", N.lib().skd_device_sm_count(dev, ctypes.byref(v)))
    return v.value


def default_ctas(shape: Optional[N.Shape] = None, device: Optional[int] = None) -> int:
    """Stream-K workers for one wave: one per SM for GQA; for absorbed MLA a
    worker is a 2-CTA cluster (a score SM and a value SM), so the number of
    such clusters the device holds at once."""
    if shape is None or shape.kind != N.SKD_KIND_MLA:
        return sm_count(device)
    dev = torch.cuda.current_device() if device is None else int(device)
    v = ctypes.c_int(0)
    N.check("skd_default_workers", N.lib().skd_default_workers(ctypes.byref(shape), dev, ctypes.byref(v)))
    return v.value


# Fixed per-segment cost of the absorbed-MLA kernel in granules of KV work:
# loading a request's 128 query rows into TMEM and draining its 128x512
# accumulator cost a few microseconds, which the dense kernel streams as
# roughly this many granules. The sparse (top-k) path gathers its rows and
# spends several times as long per granule, so the same cost is fewer
# granules there.
MLA_SEG_COST = 40
MLA_SPARSE_SEG_COST = 4


def default_seg_cost(shape: Optional[N.Shape] = None, sparse: bool = False) -> int:
    """Per-segment cost (granules) the planner charges by default: the MLA
    kernel pays a fixed cost per segment (``sparse``: plans over top-k lists),
    the GQA kernel a negligible one."""
    if shape is None or shape.kind != N.SKD_KIND_MLA:
        return 0
    return MLA_SPARSE_SEG_COST if sparse else MLA_SEG_COST


# The absorbed-MLA kernel reads a request in whole blocks of 64 tokens (4
# granules): plans for it cut only at block boundaries, so no block is read by
# two splits.
MLA_ALIGN = 4


def default_align(shape: Optional[N.Shape] = None) -> int:
    """Granules per cut unit the planner uses by default: the MLA kernel's
    64-token block, 1 (any granule) for the GQA kernel."""
    if shape is None or shape.kind != N.SKD_KIND_MLA:
        return 1
    return MLA_ALIGN


def plan_bytes(batch: int, num_kv_heads: int, n_ctas: int) -> int:
    return int(N.lib().skd_plan_bytes(batch, num_kv_heads, n_ctas))


def plan(seqlens, num_kv_heads: int, page_size: int, n_ctas: Optional[int] = None,
         mode: str = "streamk", seg_cost: int = 0, align: int = 1) -> torch.Tensor:
    """Host planner. ``seqlens``: CPU int32 tensor (or anything torch.as_tensor
    takes). ``seg_cost``: virtual granules charged per work item; ``align``:
    split points on multiples of 16 * align tokens (both Stream-K only; 0 and
    1 = the plain equal split). Returns the plan as a CPU int32 tensor; copy it
    to the device."""
    sl = torch.as_tensor(seqlens, dtype=torch.int32).contiguous()
    if sl.device.type != "cpu":
        raise ValueError("plan() takes host seqlens; use plan_device() for device seqlens")
    n = sm_count() if n_ctas is None else int(n_ctas)
    nb = plan_bytes(int(sl.numel()), num_kv_heads, n)
    if nb == 0:
        raise ValueError("invalid batch / num_kv_heads / n_ctas")
    out = torch.zeros(nb // 4, dtype=torch.int32)
    if mode == "streamk":
        N.check("skd_decode_plan_aligned", N.lib().skd_decode_plan_aligned(
            sl.data_ptr(), int(sl.numel()), int(num_kv_heads), int(page_size), n, int(seg_cost), int(align),
            out.data_ptr(), nb))
    else:
        if seg_cost or align != 1:
            raise ValueError("seg_cost and align apply to the streamk mode only")
        N.check("skd_decode_plan", N.lib().skd_decode_plan(
            sl.data_ptr(), int(sl.numel()), int(num_kv_heads), int(page_size), n, _MODES[mode],
            out.data_ptr(), nb))
    return out


def plan_device(seqlens: torch.Tensor, num_kv_heads: int, page_size: int, n_ctas: int,
                out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, seg_cost: int = 0, align: int = 1) -> torch.Tensor:
    """Device planner (graph capturable), byte-identical to ``plan``.
    ``seqlens``: CUDA int32 tensor."""
    if seqlens.device.type != "cuda" or seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous CUDA int32 tensor")
    nb = plan_bytes(int(seqlens.numel()), num_kv_heads, n_ctas)
    if out is None:
        out = torch.empty(nb // 4, dtype=torch.int32, device=seqlens.device)
    N.check("skd_decode_plan_aligned_device", N.lib().skd_decode_plan_aligned_device(
        seqlens.data_ptr(), int(seqlens.numel()), int(num_kv_heads), int(page_size), int(n_ctas),
        int(seg_cost), int(align), out.data_ptr(), out.numel() * 4, _stream_ptr(stream)))
    return out


def make_shape(q: torch.Tensor, k_pages: torch.Tensor, v_pages: Optional[torch.Tensor],
               page_table: torch.Tensor, *, scale: float, causal: bool,
               head_dim_v: Optional[int] = None) -> N.Shape:
    """skd_shape_t from tensor shapes. GQA: q [B,T,Hq,D], k/v [NP,P,Hkv,D].
    Absorbed MLA: v_pages None, k_pages [NP,P,576] or [NP,P,1,576], Dv 512."""
    B, T, Hq, Dk = (int(x) for x in q.shape)
    mla = v_pages is None
    if mla:
        NP, P = int(k_pages.shape[0]), int(k_pages.shape[1])
        Hkv, Dv, vstride = 1, int(head_dim_v or 512), Dk
    else:
        NP, P, Hkv = (int(x) for x in k_pages.shape[:3])
        Dv = int(v_pages.shape[3])
        vstride = Dv
    return N.Shape(batch=B, q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv, head_dim_qk=Dk,
                   head_dim_v=Dv, page_size=P, max_pages_per_req=int(page_table.shape[1]),
                   num_pages=NP, v_row_stride=vstride, scale=float(scale), causal=int(bool(causal)),
                   kind=N.SKD_KIND_MLA if mla else N.SKD_KIND_GQA)


def workspace(shape: N.Shape, n_ctas: int, device=None) -> torch.Tensor:
    """Allocate and zero the workspace for ``shape`` and ``n_ctas`` CTAs."""
    nb = int(N.lib().skd_workspace_bytes(ctypes.byref(shape), int(n_ctas)))
    if nb == 0:
        raise SkdError("skd_workspace_bytes", N.SKD_EUNSUPPORTED)
    ws = torch.empty(nb, dtype=torch.uint8, device=device or "cuda")
    N.check("skd_workspace_reset", N.lib().skd_workspace_reset(ws.data_ptr(), nb, _stream_ptr(None)))
    return ws


def _chk(t: torch.Tensor, name: str, dtype):
    if t.device.type != "cuda" or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def decode_attention(q, k_pages, v_pages, page_table, seqlens, plan_dev, ws, *, scale: float,
                     causal: Optional[bool] = None, n_ctas: Optional[int] = None,
                     out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     shape: Optional[N.Shape] = None,
                     stream: Optional[torch.cuda.Stream] = None,
                     two_kernel: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Enqueue one decode-attention launch; returns (out bf16 [B,T,Hq,Dv], lse fp32 [B,T,Hq]).
    ``two_kernel``: the split-KV comparator (splits write partial states, a
    second kernel merges them); meant for plans of mode "fixed_split"."""
    _chk(q, "q", torch.bfloat16)
    _chk(k_pages, "k_pages", torch.bfloat16)
    if v_pages is not None:
        _chk(v_pages, "v_pages", torch.bfloat16)
    _chk(page_table, "page_table", torch.int32)
    _chk(seqlens, "seqlens", torch.int32)
    _chk(plan_dev, "plan", torch.int32)
    if causal is None:
        causal = q.shape[1] > 1
    if shape is None:
        shape = make_shape(q, k_pages, v_pages, page_table, scale=scale, causal=causal)
    B, T, Hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    if out is None:
        out = torch.empty(B, T, Hq, shape.head_dim_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, Hq, dtype=torch.float32, device=q.device)
    n = int(plan_dev[3].item()) if n_ctas is None else int(n_ctas)
    vp = k_pages if v_pages is None else v_pages
    fn = "skd_decode_attention_split_combine" if two_kernel else "skd_decode_attention"
    N.check(fn, getattr(N.lib(), fn)(
        ctypes.byref(shape), q.data_ptr(), k_pages.data_ptr(), vp.data_ptr(), page_table.data_ptr(),
        seqlens.data_ptr(), plan_dev.data_ptr(), n, ws.data_ptr(), ws.numel(), out.data_ptr(),
        lse.data_ptr(), _stream_ptr(stream)))
    return out, lse


def decode_attention_sparse(q, kv_pages, page_table, seqlens, topk_idx, topk_len, plan_dev, ws, *,
                            scale: float, n_ctas: Optional[int] = None,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            shape: Optional[N.Shape] = None,
                            stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse (top-k) absorbed-MLA decode: request b attends only to the cache
    positions ``topk_idx[b, :topk_len[b]]`` (int32 [B, K] and [B] on the
    device). ``plan_dev`` must come from the planner run over ``topk_len``
    (``plan(topk_len_host, 1, page_size, n)``). Returns (out, lse) like
    ``decode_attention``."""
    _chk(q, "q", torch.bfloat16)
    _chk(kv_pages, "kv_pages", torch.bfloat16)
    _chk(page_table, "page_table", torch.int32)
    _chk(seqlens, "seqlens", torch.int32)
    _chk(topk_idx, "topk_idx", torch.int32)
    _chk(topk_len, "topk_len", torch.int32)
    _chk(plan_dev, "plan", torch.int32)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != q.shape[0] or topk_len.numel() != q.shape[0]:
        raise ValueError("topk_idx must be [B, K] and topk_len [B]")
    if shape is None:
        shape = make_shape(q, kv_pages, None, page_table, scale=scale, causal=False)
    B, T, Hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    if out is None:
        out = torch.empty(B, T, Hq, shape.head_dim_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, Hq, dtype=torch.float32, device=q.device)
    n = int(plan_dev[3].item()) if n_ctas is None else int(n_ctas)
    N.check("skd_decode_attention_sparse", N.lib().skd_decode_attention_sparse(
        ctypes.byref(shape), q.data_ptr(), kv_pages.data_ptr(), page_table.data_ptr(), seqlens.data_ptr(),
        topk_idx.data_ptr(), int(topk_idx.shape[1]), topk_len.data_ptr(), plan_dev.data_ptr(), n,
        ws.data_ptr(), ws.numel(), out.data_ptr(), lse.data_ptr(), _stream_ptr(stream)))
    return out, lse


def set_pdl(enable: bool) -> None:
    """Launch the attention kernel with programmatic dependent launch (default
    on): it may be scheduled while the previous kernel of the stream, e.g. the
    device planner, is still running, and waits for it before reading inputs."""
    N.check("skd_set_pdl", N.lib().skd_set_pdl(1 if enable else 0))


def read_error(ws: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    v = ctypes.c_int32(0)
    N.check("skd_read_error", N.lib().skd_read_error(ws.data_ptr(), ctypes.byref(v), _stream_ptr(stream)))
    return int(v.value)
