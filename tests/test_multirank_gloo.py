"""Multi-rank paths on CPU with the gloo backend (world size 2).

(A) batch sharding: each rank decodes its shard, no collective on the data
    path; the gathered rows must equal the single-process result exactly.
(C) one long request split by key range across ranks: partial states are
    exchanged with all_gather and merged; the result must equal the unsplit
    attention.
Rank arithmetic uses the fp64 oracle (no GPU here); what is tested is the host
logic of sharding.py and the exchange pattern.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W
from oracle import attention as A
from sm_load_balancing_gb300 import sharding as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _sub_workload(w, idx):
    """The requests `idx` of w as a workload of their own (same cache)."""
    sub = W.make_custom([1], num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                        head_dim_qk=w.head_dim_qk, page_size=w.page_size, q_tokens=w.q_tokens,
                        causal=w.causal, scale=w.scale)
    sub.batch = len(idx)
    sub.seqlens = np.ascontiguousarray(w.seqlens[idx])
    sub.page_table = np.ascontiguousarray(w.page_table[idx])
    sub.q = np.ascontiguousarray(w.q[idx])
    sub.k_pages, sub.v_pages = w.k_pages, w.v_pages
    return sub


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # ---- (A) batch sharding, no collective on the data path ----
        w = W.make_custom([5, 900, 33, 0, 260, 1200, 17], num_q_heads=8, num_kv_heads=2,
                          head_dim_qk=32, page_size=16, seed=3)
        shards = S.shard_batch(w.seqlens, world)
        mine = shards[rank]
        out, lse = A.decode_workload(_sub_workload(w, mine)) if len(mine) else (None, None)
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine.tolist(), out, lse))   # test-side assembly only
        # ---- (C) one request split by key range, one exchange + merge ----
        wl = W.make_custom([1000], num_q_heads=4, num_kv_heads=1, head_dim_qk=32, seed=4)
        lo, hi = S.split_keys(1000, world)[rank]
        k, v = A.gather_rows(wl, 0, 0, 1000)
        qs = [W.bf16_bits_to_fp32(wl.q[0, 0, h]).astype(np.float64) for h in range(4)]
        parts = [A.partial_state(qs[h], k[lo:hi], v[lo:hi], wl.scale) for h in range(4)]
        allparts = [None] * world
        dist.all_gather_object(allparts, parts)
        merged = [A.merge_states([allparts[r][h] for r in range(world)]) for h in range(4)]
        if rank == 0:
            q.put(("ok", gathered, merged))
    except Exception as e:  # report to the parent instead of hanging it
        q.put(("err", repr(e), None))
    finally:
        dist.destroy_process_group()


def test_sharding_rules():
    sh = S.shard_batch([5, 900, 33, 0, 260, 1200, 17], 2)
    assert sorted(np.concatenate(sh).tolist()) == list(range(7))
    loads = [sum([5, 900, 33, 0, 260, 1200, 17][i] for i in s) for s in sh]
    assert abs(loads[0] - loads[1]) <= 1200
    assert S.split_keys(1000, 2) == [(0, 496), (496, 1000)]
    assert S.split_keys(10, 3) == [(0, 0), (0, 0), (0, 10)]


def test_two_ranks_gloo_batch_shard_and_key_split():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        status, gathered, merged = q.get(timeout=240)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert status == "ok", gathered
    w = W.make_custom([5, 900, 33, 0, 260, 1200, 17], num_q_heads=8, num_kv_heads=2,
                      head_dim_qk=32, page_size=16, seed=3)
    ref_out, ref_lse = A.decode_workload(w)
    seen = set()
    for idx, out, lse in gathered:
        for j, b in enumerate(idx):
            assert b not in seen
            seen.add(b)
            np.testing.assert_array_equal(out[j], ref_out[b])
            np.testing.assert_array_equal(lse[j], ref_lse[b])
    assert seen == set(range(7))
    wl = W.make_custom([1000], num_q_heads=4, num_kv_heads=1, head_dim_qk=32, seed=4)
    ro, rl = A.decode_workload(wl)
    for h in range(4):
        np.testing.assert_allclose(merged[h][0], ro[0, 0, h], rtol=0, atol=1e-12)
        assert merged[h][1] == pytest.approx(rl[0, 0, h], abs=1e-12)
