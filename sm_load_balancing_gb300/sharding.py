"""Host-side sharding of a decode batch across GPUs (one process per GPU).

The decode path partitions naturally: every (request, kv-head group) item is
independent, so a batch is sharded by requests with no collective on the data
path; each rank runs the single-GPU Stream-K kernel on its shard and writes its
own rows of out/lse.

A request too long for one GPU can be split by key range; the ranks then hold
partial softmax states of the same rows and need one exchange followed by the
merge of partial states ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）",
core method: reduce the partial outputs of split-KV attention), the same
reduction the kernel performs across CTAs.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

GRANULE = 16


def shard_batch(seqlens: Sequence[int], world_size: int) -> List[np.ndarray]:
    """Longest-processing-time assignment of requests to ranks.

    Requests are taken in decreasing length (ties: lower index first) and each
    goes to the rank with the least KV tokens so far (ties: lower rank). Every
    request lands on exactly one rank; returns the sorted request indices of
    each rank."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    L = np.asarray(seqlens, dtype=np.int64)
    order = sorted(range(len(L)), key=lambda i: (-int(L[i]), i))
    load = [0] * world_size
    owned: List[List[int]] = [[] for _ in range(world_size)]
    for i in order:
        r = min(range(world_size), key=lambda k: (load[k], k))
        owned[r].append(i)
        load[r] += int(L[i])
    return [np.array(sorted(o), dtype=np.int64) for o in owned]


def split_keys(seqlen: int, world_size: int, granule: int = GRANULE) -> List[Tuple[int, int]]:
    """Key ranges [lo, hi) of one request for each rank: the request's granules
    cut into world_size near-equal contiguous chunks (the one-wave equal split,
    applied across GPUs)."""
    g = -(-int(seqlen) // granule)
    out = []
    for r in range(world_size):
        lo = (r * g) // world_size * granule
        hi = min(((r + 1) * g) // world_size * granule, int(seqlen))
        out.append((min(lo, int(seqlen)), hi))
    return out
