#!/usr/bin/env python3
"""Decode-attention benchmark: µs per call and achieved HBM TB/s on one GB300.

A step is one decode-attention call over the whole batch of the workload (the
Stream-K plan + one persistent kernel). Default workload: the Llama-3-8B-shaped
GQA decode batch (B=32, 32 q / 8 kv heads, D=128, L ~ U[512, 8192], P=16).

  value   algorithmic bytes / device time (CUDA events on the launching stream),
          inputs resident in HBM; when a step reads less than twice L2's size a
          256 MB write evicts L2 before every step (each step then has its own
          events), otherwise the steps run back to back between two events
  e2e     the same metric through the public API with host buffers, KV cache
          resident: for Stream-K plans DecodeStep.run() (one graph replay of the
          pinned H2D copies of q / page table / seqlens, the device planner, the
          kernel and the D2H copies of out / lse, then a host wait); otherwise
          the eager calls with the host planner and the plan copied too
  roofline  achieved = algorithmic bytes / mean kernel time against the measured
          HBM copy bandwidth (MEASURED_PEAKS.json, else a 6.8 TB/s fallback);
          traffic = ncu DRAM bytes per launch recorded in profiles/, reported
          only while the kernel source hash matches the one captured
  cpu_baseline  the fp64 oracle on a bounded sample, on all host cores
  clocks  nvidia-smi samples taken during the timed region

--impl reference times the fp64 CPU oracle on the host cores instead.
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling, no
collective on the data path); value = all ranks' bytes / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/call and achieved HBM TB/s (% of roofline) on 1 GB300"
L2_BYTES = 129 * 1000 * 1000
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = {"gqa": "sm_load_balancing_gb300/csrc/gqa_decode.cu",
              "mla": "sm_load_balancing_gb300/csrc/mla_decode.cu"}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_gqa")
    ap.add_argument("--mode", choices=["streamk", "round_robin", "fixed_split"], default="streamk",
                    help="fixed_split = the two-kernel split-KV comparator (fixed splits + combine kernel)")
    ap.add_argument("--seg-cost", type=int, default=None,
                    help="planner's per-segment cost in granules (default: the library's per-kind default)")
    ap.add_argument("--align", type=int, default=None,
                    help="planner's cut unit in granules (default: the library's per-kind default)")
    ap.add_argument("--n-ctas", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--launch-study", action="store_true",
                    help="also time one step = device planner + attention: eager vs CUDA graph, "
                         "with and without programmatic dependent launch")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"

    def find(o):
        if isinstance(o, dict):
            for k, v in o.items():
                if k.lower() in ("hbm_gbs", "hbm_gb_s", "hbm_bandwidth_gbs") and isinstance(v, (int, float)):
                    return float(v)
                r = find(v)
                if r:
                    return r
        return None
    v = find(d)
    return (v, "measured (MEASURED_PEAKS.json hbm_gbs)") if v else (FALLBACK_HBM_GBS, "fallback")


def _launch_study(skd, q, k, v, pt, sl, w, shape, n, seg_cost, align, ws, out, lse, a):
    """Per-step time of device planner + attention, four ways: eager launches or
    one CUDA graph replay, each with programmatic dependent launch on or off.
    The difference to the kernel time alone is what launching costs per step."""
    import torch
    hkv = shape.num_kv_heads
    plan = skd.plan_device(sl, hkv, w.page_size, n, seg_cost=seg_cost, align=align)
    res = {}
    steps = max(50, min(a.steps, 500))
    for pdl in (False, True):
        skd.set_pdl(pdl)

        def step():
            skd.plan_device(sl, hkv, w.page_size, n, out=plan, seg_cost=seg_cost, align=align)
            skd.decode_attention(q, k, v, pt, sl, plan, ws, scale=w.scale, causal=w.causal, n_ctas=n,
                                 out=out, lse=lse, shape=shape)

        for _ in range(5):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=st):
            step()
        torch.cuda.current_stream().wait_stream(st)
        for name, fn in (("eager", step), ("graph", g.replay)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            res[f"{name}{'_pdl' if pdl else ''}_us"] = e0.elapsed_time(e1) / steps * 1e3
    skd.set_pdl(True)
    if skd.read_error(ws) != 0:
        raise RuntimeError(f"device error word {skd.read_error(ws)}")
    res["steps"] = steps
    return res


def _traffic(kind, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    src = os.path.join(ROOT, KERNEL_SRC[kind])
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        e = d.get(workload)
        if e and e.get("kernel_src_sha256_16") == sha:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi sampler for the SM clock and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def _cpu_oracle_sample(w, target_s):
    """Time the fp64 oracle on the first requests of the batch, about
    `target_s` seconds of work. Returns (bytes_per_s, cores, description)."""
    import numpy as np

    from oracle import attention as A
    A.build()
    rows_per_req = w.q_tokens * w.num_q_heads
    decode = A.decode_sparse_workload if w.sparse else A.decode_workload
    lens = w.topk_len if w.sparse else w.seqlens  # KV rows each request reads
    # probe one request to size the sample
    order = list(range(w.batch))
    t0 = time.perf_counter()
    decode(w, rows=list(range(rows_per_req)))
    per_req = max(time.perf_counter() - t0, 1e-4) / max(int(lens[0]), 1)
    budget_tokens = target_s / per_req
    chosen, toks = [], 0
    for b in order:
        if chosen and toks + int(lens[b]) > budget_tokens:
            break
        chosen.append(b)
        toks += int(lens[b])
    rows = [b * rows_per_req + r for b in chosen for r in range(rows_per_req)]
    # repeat a short sample until it has run for a few seconds (stable timing)
    reps, dt = 0, 0.0
    while reps == 0 or (dt < min(3.0, target_s) and reps < 1000):
        t0 = time.perf_counter()
        decode(w, rows=rows)
        dt += time.perf_counter() - t0
        reps += 1
    frac = toks / max(w.kv_tokens, 1)
    sample_bytes = w.algorithmic_bytes() * frac * reps
    desc = (f"all {rows_per_req} query rows of requests 0..{chosen[-1]} "
            f"({len(chosen)} of {w.batch} requests, {toks} of {w.kv_tokens} KV tokens), "
            f"{reps} repetition(s), fp64 C oracle{' (sparse)' if w.sparse else ''}, OpenMP")
    return sample_bytes / dt, A.num_threads(), desc, dt


def run_reference(a):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import workloads as W
    w = W.make(a.workload)
    from oracle import attention as A
    A.build()
    # each step: a bounded sample of the workload (same rows every step)
    per_step = max(0.5, min(10.0, 150.0 / max(a.steps + a.warmup, 1)))
    for _ in range(a.warmup):
        _cpu_oracle_sample(w, per_step * 0.2)
    vals, times = [], []
    desc, cores = "", 1
    for _ in range(a.steps):
        v, cores, desc, dt = _cpu_oracle_sample(w, per_step)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1e3 * w.algorithmic_bytes() / (value * 1e12),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16, random page permutation)",
        "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "workload"},
                   "l2": "CPU run"},
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def run_ours(a):
    import numpy as np
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import sm_load_balancing_gb300 as skd
    import workloads as W

    w = W.make(a.workload, seed=rank)
    kind = "mla" if w.mla else "gqa"

    def bf16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)

    q = bf16(w.q).to(dev)
    k = bf16(w.k_pages).to(dev)
    v = None if w.mla else bf16(w.v_pages).to(dev)
    pt = torch.from_numpy(w.page_table).to(dev)
    sl = torch.from_numpy(w.seqlens).to(dev)
    sparse = w.sparse
    if sparse:
        if a.mode == "fixed_split":
            raise SystemExit("the two-kernel comparator is not built for the sparse path")
        ti = torch.from_numpy(w.topk_idx).to(dev)
        tl = torch.from_numpy(w.topk_len).to(dev)
    plan_lens = w.topk_len if sparse else w.seqlens  # the planner splits what each request reads
    shape = skd.make_shape(q, k, v, pt, scale=w.scale, causal=w.causal)
    n = a.n_ctas or skd.default_ctas(shape)
    seg_cost = 0 if a.mode != "streamk" else (skd.default_seg_cost(shape, sparse=sparse) if a.seg_cost is None
                                              else a.seg_cost)
    align = 1 if a.mode != "streamk" else (skd.default_align(shape) if a.align is None else a.align)
    plan_h = skd.plan(plan_lens, shape.num_kv_heads, w.page_size, n, a.mode, seg_cost=seg_cost, align=align)
    plan_d = plan_h.to(dev)
    ws = skd.workspace(shape, n, dev)
    out = torch.empty(w.batch, w.q_tokens, w.num_q_heads, w.head_dim_v, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.batch, w.q_tokens, w.num_q_heads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    two_kernel = a.mode == "fixed_split"

    prefix = None
    if w.prefix_groups:
        # shared-prefix decode: prefix pass + suffix pass + merge (4 launches of ours per step)
        from sm_load_balancing_gb300.prefix import SharedPrefixDecode
        if a.mode != "streamk" or sparse:
            raise SystemExit("shared-prefix decode runs the Stream-K plans only")
        prefix = SharedPrefixDecode(q, k, v, w.page_table, w.seqlens, w.prefix_groups, w.prefix_lens,
                                    scale=w.scale, causal=w.causal, n_ctas=n)

    def step():
        if prefix is not None:
            prefix(q, out=out, lse=lse, stream=stream)
        elif sparse:
            skd.decode_attention_sparse(q, k, pt, sl, ti, tl, plan_d, ws, scale=w.scale, n_ctas=n, out=out,
                                        lse=lse, shape=shape, stream=stream)
        else:
            skd.decode_attention(q, k, v, pt, sl, plan_d, ws, scale=w.scale, causal=w.causal, n_ctas=n,
                                 out=out, lse=lse, shape=shape, stream=stream, two_kernel=two_kernel)

    # bytes a step reads: when they are under twice L2 (129 MB), part of them could
    # still be in L2 from the previous step, so a 256 MB write evicts it before
    # every timed step (outside the per-step events)
    flush = None
    if w.algorithmic_bytes() < 2 * L2_BYTES:
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    if skd.read_error(ws) != 0:
        raise RuntimeError(f"device error word {skd.read_error(ws)}")
    # Without a flush the K steps run back to back between two events on the
    # launching stream (an event between launches would add a gap of its own);
    # with a flush, each step has its own pair of events so that the flush
    # writes stay outside the measured steps.
    ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
          if flush is not None else [])
    barrier()
    torch.cuda.synchronize()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(a.steps):
        if flush is not None:
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        else:
            step()
    t_all1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ck = clocks.stop()
    total_ms = t_all0.elapsed_time(t_all1)
    per = [s.elapsed_time(e) for s, e in ev] if ev else [total_ms / a.steps]
    mean_kernel_ms = sum(per) / len(per)
    err = skd.read_error(ws)
    if err != 0:
        raise RuntimeError(f"device error word {err}")
    launch = _launch_study(skd, q, k, v, pt, sl, w, shape, n, seg_cost, align, ws, out, lse, a) if a.launch_study else None
    if prefix is not None:
        for wsx in prefix.workspaces():
            if skd.read_error(wsx) != 0:
                raise RuntimeError(f"device error word {skd.read_error(wsx)}")
        # context: the plain decode of the full sequences reads every prefix once per request
        ref_us = []
        for _ in range(max(3, min(a.steps, 50))):
            if flush is not None:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            skd.decode_attention(q, k, v, pt, sl, plan_d, ws, scale=w.scale, causal=w.causal, n_ctas=n,
                                 out=out, lse=lse, shape=shape, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ref_us.append(e0.elapsed_time(e1) * 1e3)
        prefix_ctx = {"plain_decode_us": statistics.median(ref_us[2:] or ref_us),
                      "plain_decode_kv_tokens": int(w.seqlens.astype("int64").sum()),
                      "virtual_prefix_requests": prefix.V, "requests_per_virtual": prefix.R}

    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms, mean_kernel_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms, mean_kernel_ms = float(t[0].item()), float(t[1].item())

    alg_bytes = w.algorithmic_bytes()
    # with flushes in the loop a step is its own event span, else the whole loop / steps
    ms_per_step = (mean_kernel_ms if flush is not None else total_ms / a.steps)
    value = world * alg_bytes / (ms_per_step * 1e-3) / 1e12  # TB/s, all ranks

    # ---- e2e through the public API with host buffers ----
    e2e = None
    if not a.no_e2e:
        q_h = bf16(w.q).pin_memory()
        pt_h = torch.from_numpy(w.page_table).pin_memory()
        sl_h = torch.from_numpy(w.seqlens).pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        q_d, pt_d, sl_d = torch.empty_like(q), torch.empty_like(pt), torch.empty_like(sl)
        plan_pin = torch.empty_like(plan_h).pin_memory()
        plan_dd = torch.empty_like(plan_d)
        if sparse:
            ti_h = torch.from_numpy(w.topk_idx).pin_memory()
            tl_h = torch.from_numpy(w.topk_len).pin_memory()
            ti_d, tl_d = torch.empty_like(ti), torch.empty_like(tl)

        # the serving-loop API: one captured step (H2D, device planner, decode, D2H)
        step = None
        if prefix is None and a.mode == "streamk":
            from sm_load_balancing_gb300.step import DecodeStep
            step = DecodeStep(q, k, v, w.page_table.shape[1], scale=w.scale, causal=w.causal,
                              topk=int(w.topk_idx.shape[1]) if sparse else None, n_ctas=n, seg_cost=seg_cost,
                              align=align)
            step.q_host.copy_(q_h)
            step.page_table_host.copy_(pt_h)
            step.seqlens_host.copy_(sl_h)
            if sparse:
                step.topk_idx_host.copy_(ti_h)
                step.topk_len_host.copy_(tl_h)

        def e2e_step():
            if step is not None:
                step.run()
                return
            lens_h = tl_h if sparse else sl_h
            p = skd.plan(lens_h, shape.num_kv_heads, w.page_size, n, a.mode, seg_cost=seg_cost,
                         align=align)  # host planner
            plan_pin.copy_(p)
            q_d.copy_(q_h, non_blocking=True)
            pt_d.copy_(pt_h, non_blocking=True)
            sl_d.copy_(sl_h, non_blocking=True)
            plan_dd.copy_(plan_pin, non_blocking=True)
            if prefix is not None:
                prefix(q_d, out=out, lse=lse, stream=stream)
            elif sparse:
                ti_d.copy_(ti_h, non_blocking=True)
                tl_d.copy_(tl_h, non_blocking=True)
                skd.decode_attention_sparse(q_d, k, pt_d, sl_d, ti_d, tl_d, plan_dd, ws, scale=w.scale, n_ctas=n,
                                            out=out, lse=lse, shape=shape, stream=stream)
            else:
                skd.decode_attention(q_d, k, v, pt_d, sl_d, plan_dd, ws, scale=w.scale, causal=w.causal,
                                     n_ctas=n, out=out, lse=lse, shape=shape, stream=stream, two_kernel=two_kernel)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(a.warmup):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        n_e2e = max(1, min(a.steps, 500))
        for _ in range(n_e2e):
            e2e_step()
        t_e2e = (time.perf_counter() - t0) / n_e2e
        barrier()
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([t_e2e], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            t_e2e = float(t.item())
        if step is not None:
            h2d, d2h = step.host_to_device_bytes(), step.device_to_host_bytes()
            note = ("DecodeStep.run(): one CUDA graph replay of pinned H2D of q/page table/seqlens"
                    + ("/top-k lists" if sparse else "") + " + device planner + kernel + D2H of out/lse, "
                    "then a host wait; KV cache resident")
        else:
            h2d = q_h.numel() * 2 + pt_h.numel() * 4 + sl_h.numel() * 4 + plan_pin.numel() * 4
            if sparse:
                h2d += ti_h.numel() * 4 + tl_h.numel() * 4
            d2h = out_h.numel() * 2 + lse_h.numel() * 4
            note = ("host planner + pinned H2D of q/seqlens/page table/plan" + ("/top-k lists" if sparse else "")
                    + " + kernel + D2H of out/lse; KV cache resident"
                    + ("; shared prefix: its layouts and plans are prepared once, outside the loop"
                       if prefix is not None else ""))
        e2e = {"value": world * alg_bytes / t_e2e / 1e12, "unit": "TB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "us_per_step": t_e2e * 1e6, "steps": n_e2e, "note": note}
        if skd.read_error(ws) != 0 or (step is not None and step.error() != 0):
            raise RuntimeError("device error in e2e loop")

    peak, peak_src = _measured_hbm_peak()
    achieved = alg_bytes / (mean_kernel_ms * 1e-3) / 1e9
    traffic = _traffic(kind, w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_per_step, "us_per_call": ms_per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, random page permutation)",
        "config": {"workload": w.name, **{kk: vv for kk, vv in w.describe().items() if kk != "workload"},
                   "n_ctas": n, "plan": a.mode, "seg_cost": seg_cost, "align": align, "algorithmic_bytes": alg_bytes,
                   "l2": ("flushed before each timed step (256 MB write, outside the step's events)"
                          if flush is not None else "no flush: KV per step is larger than L2 (129 MB)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": f"{kind}_decode_kernel", "launch_ms_mean": mean_kernel_ms,
                     "launch_ms_median": statistics.median(per),
                     "launch_timing": ("per-step events around each launch (flush between steps)" if ev else
                                       "back-to-back launches: timed region / steps")},
        "e2e": e2e,
        "gpu_launches": a.steps * (prefix.launches() if prefix is not None else 2 if two_kernel else 1),
        "clocks": ck,
    }
    if launch is not None:
        line["launch"] = launch
    if prefix is not None:
        line["shared_prefix"] = prefix_ctx
        line["roofline"]["kernel"] = ("shared-prefix step (gather + gqa_decode + merge)" if prefix.fused else
                                      "shared-prefix step (gqa_decode x2 + gather + merge)")
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        try:
            bps, cores, desc, dt = _cpu_oracle_sample(w, a.cpu_seconds)
            line["cpu_baseline"] = {"value": bps / 1e12, "unit": "TB/s", "cores": cores,
                                    "kind": "oracle", "sample": desc, "seconds": dt}
        except Exception as ex:  # the bench line must still print
            line["cpu_baseline"] = {"value": None, "unit": "TB/s", "cores": None, "kind": "oracle",
                                    "sample": f"failed: {ex}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    a = _args()
    if a.impl == "reference":
        return run_reference(a)
    return run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
