"""Work-split definitions (TEST INFRASTRUCTURE; see the package docstring).

All integer arithmetic, so the CUDA library's planners must agree with these
bit for bit.

streamk_split
    "传统 GEMM 计算可能因任务大小不均产生多个调度波次（Waves）..." (triton.csdn.net
    Q&A on waves and FlashMLA's Stream-K), closing summary: cut the total work
    into exactly as many near-equal chunks as there are SMs and launch a single
    wave. Here the work is the batch's KV tokens, counted per (request, kv head)
    work item in granules of ``granule`` tokens; chunk c is the granule range
    [floor(c*G/n), floor((c+1)*G/n)) of the concatenation of all items in
    (request, kv head) order, and each chunk is cut at item boundaries into
    segments. "MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", core method:
    the split is decided at run time from the real sequence lengths.

    Optional ``seg_cost`` (an extension; the pages charge nothing per
    segment): each non-empty item is preceded by ``seg_cost`` virtual granules
    that hold no tokens, so the equal split runs over tokens plus a fixed cost
    per item start. ``seg_cost = 0`` is the split above.

round_robin_split
    Whole work items dealt to workers in turn, the way the GLM-5.2 decode
    article ("GLM-5.2-FP8 ... B300", MegaRTP KernelPlan paragraph) deals tile
    tasks to worker queues. It is the unbalanced comparator.

fixed_split
    The two-kernel split-KV comparator: a fixed number of splits per item,
    merged afterwards by a separate combine step.

round_robin_queues / list_schedule
    The two worked examples the pages print: the MegaRTP queue fill
    (732 tasks over 148 queues) and the 4-SM / 8-task timeline of the Q&A page.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def streamk_split(seqlens: Sequence[int], num_kv_heads: int, n_ctas: int,
                  granule: int = 16, seg_cost: int = 0) -> Dict:
    """Stream-K one-wave split.

    Returns a dict with
      segments:  list per CTA of tuples (item, tok_begin, tok_end)
      item_splits: list per item of [(cta, tok_begin, tok_end)] in split order
      bounds:    granule boundaries floor(c*G/n), c = 0..n
      total_granules: G
    Items are i = b * num_kv_heads + h, of length seqlens[b] tokens. An item of
    length 0 occupies no work; it is a segment of the first CTA whose chunk ends
    after its position (the last CTA if none).
    """
    if n_ctas <= 0 or num_kv_heads <= 0 or granule <= 0 or seg_cost < 0:
        raise ValueError("n_ctas, num_kv_heads and granule must be positive, seg_cost >= 0")
    L = [int(x) for x in seqlens]
    items = [(b * num_kv_heads + h, L[b]) for b in range(len(L)) for h in range(num_kv_heads)]
    starts = []
    pos = 0
    for _, length in items:
        if length > 0:
            pos += seg_cost  # the item's virtual start cost, before its tokens
        starts.append(pos)
        pos += _ceil_div(length, granule)
    total = pos
    bounds = [(c * total) // n_ctas for c in range(n_ctas + 1)]
    segments: List[List[Tuple[int, int, int]]] = [[] for _ in range(n_ctas)]
    item_splits: List[List[Tuple[int, int, int]]] = [[] for _ in items]
    for (i, length), s in zip(items, starts):
        e = s + _ceil_div(length, granule)
        if e == s:
            owner = next((c for c in range(n_ctas) if bounds[c + 1] > s), n_ctas - 1)
            segments[owner].append((i, 0, 0))
            item_splits[i].append((owner, 0, 0))
            continue
        for c in range(n_ctas):
            lo, hi = max(s, bounds[c]), min(e, bounds[c + 1])
            if lo < hi:
                tb = (lo - s) * granule
                te = min((hi - s) * granule, length)
                segments[c].append((i, tb, te))
                item_splits[i].append((c, tb, te))
    return dict(segments=segments, item_splits=item_splits, bounds=bounds,
                total_granules=total, granule=granule)


def round_robin_split(seqlens: Sequence[int], num_kv_heads: int, n_ctas: int) -> Dict:
    """Whole items dealt in turn: item i goes to CTA i mod n (no splits)."""
    L = [int(x) for x in seqlens]
    n_items = len(L) * num_kv_heads
    segments: List[List[Tuple[int, int, int]]] = [[] for _ in range(n_ctas)]
    item_splits = []
    for i in range(n_items):
        c = i % n_ctas
        segments[c].append((i, 0, L[i // num_kv_heads]))
        item_splits.append([(c, 0, L[i // num_kv_heads])])
    return dict(segments=segments, item_splits=item_splits)


def fixed_split(seqlens: Sequence[int], num_kv_heads: int, n_ctas: int, granule: int = 16) -> Dict:
    """The two-kernel comparator's split (FlashDecoding-style split-KV, which
    the pages measure MeldKernel against): every item is cut into
    S = max(1, n_ctas // n_items) near-equal granule ranges (fewer if it has
    fewer granules; one empty range if it has none); the ranges, listed in
    (item, split) order, are dealt to CTAs in turn."""
    L = [int(x) for x in seqlens]
    items = [(b * num_kv_heads + h, L[b]) for b in range(len(L)) for h in range(num_kv_heads)]
    S = max(1, n_ctas // len(items)) if items else 1
    flat = []
    item_splits: List[List[Tuple[int, int]]] = []
    for i, length in items:
        g = _ceil_div(length, granule)
        s = max(1, min(S, g))
        parts = []
        for k in range(s):
            lo, hi = (k * g) // s, ((k + 1) * g) // s
            parts.append((lo * granule, min(hi * granule, length)))
        item_splits.append(parts)
        flat += [(i, tb, te) for tb, te in parts]
    segments: List[List[Tuple[int, int, int]]] = [[] for _ in range(n_ctas)]
    for j, seg in enumerate(flat):
        segments[j % n_ctas].append(seg)
    return dict(segments=segments, item_splits=item_splits, splits_per_item=S)


def round_robin_queues(n_tasks: int, n_queues: int, pad: int = -1) -> np.ndarray:
    """Task ids dealt round-robin to queues, padded with ``pad`` (a NoOp) to a
    rectangular [n_queues, max_len] array."""
    depth = _ceil_div(n_tasks, n_queues) if n_tasks else 0
    q = np.full((n_queues, depth), pad, dtype=np.int64)
    for t in range(n_tasks):
        q[t % n_queues, t // n_queues] = t
    return q


def list_schedule(task_times: Sequence[float], n_workers: int) -> Dict:
    """Greedy dispatch: each task, in order, starts on the worker that frees up
    first (lowest index on ties). Returns per-task (worker, start, end), per-
    worker finish time, the makespan and each worker's idle time before the
    makespan."""
    free = [0.0] * n_workers
    tasks = []
    for t in task_times:
        w = min(range(n_workers), key=lambda k: (free[k], k))
        start = free[w]
        free[w] = start + t
        tasks.append((w, start, free[w]))
    makespan = max(free) if free else 0.0
    return dict(tasks=tasks, finish=free, makespan=makespan,
                idle=[makespan - f for f in free])


def streamk_loads(task_times: Sequence[int], n_workers: int) -> List[int]:
    """Per-worker load when the summed integer work is cut into n near-equal
    contiguous chunks (the one-wave split applied to a task list)."""
    total = int(sum(task_times))
    b = [(c * total) // n_workers for c in range(n_workers + 1)]
    return [b[c + 1] - b[c] for c in range(n_workers)]
