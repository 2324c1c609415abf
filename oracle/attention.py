"""fp64 attention oracle (TEST INFRASTRUCTURE; see the package docstring).

``decode`` wraps the C routine in ``oracle_decode.c``: plain softmax attention
written from its definition ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解",
section 6.3 and Q8: QK^T -> mask -> softmax -> xV).

``decode_sparse`` wraps the sparse (top-k) routine of the same file: the same
attention restricted to the cache positions each request lists (the GLM-5.2-FP8
decode article, tahou.com: the layer continues with TopK and Sparse FlashMLA,
whose ranks gather the KV rows named by the top-2048 indices).

``partial_state`` and ``merge_states`` give the split-KV view of the same
result ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", key observations and
core method): each split of the keys yields a partial state (m, l, acc) and the
reduction of all partial states is the unsplit attention. They are written in
numpy, independently of the C routine, over explicit key/value rows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_decode.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP). Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = lib.oracle_decode_f64
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int] * 10 + [ctypes.c_double] + [ctypes.c_void_p] * 3 + [
            ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p]
        f = lib.oracle_decode_sparse_f64
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int] * 9 + [ctypes.c_double] + [ctypes.c_void_p] * 3 + [
            ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


class OracleInputError(ValueError):
    pass


_ERRORS = {-1: "bad shape argument", -2: "seqlen out of range",
           -3: "page id out of range", -4: "causal with 0 < seqlen < q_tokens",
           -5: "topk_len out of range", -6: "top-k position out of range"}


def decode(*, q, k_pages, v_pages, page_table, seqlens, num_q_heads, num_kv_heads,
           head_dim_qk, head_dim_v, page_size, causal, scale, num_pages=None,
           v_row_stride=None, rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention for every (b, t, h) row, or only for ``rows``.

    q: uint16 bf16 bits [B][T][Hq][Dk]; k_pages [NP][P][Hkv][Dk];
    v_pages: [NP][P][Hkv][Dv] or None for the absorbed-MLA layout (V = the
    first Dv columns of each K row). Returns (out fp64 [n][Dv], lse fp64 [n]),
    in the shape [B][T][Hq][Dv] / [B][T][Hq] when ``rows`` is None.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k_pages, dtype=np.uint16)
    if v_pages is None:
        v = k
        vstride = head_dim_qk if v_row_stride is None else v_row_stride
    else:
        v = np.ascontiguousarray(v_pages, dtype=np.uint16)
        vstride = head_dim_v if v_row_stride is None else v_row_stride
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    B, T = int(q.shape[0]), int(q.shape[1])
    NP = int(k.shape[0]) if num_pages is None else int(num_pages)
    if rows is None:
        n = B * T * num_q_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = int(rows_arr.shape[0])
    out = np.zeros((max(n, 1), head_dim_v), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    rc = lib.oracle_decode_f64(
        B, T, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, page_size, int(pt.shape[1]),
        NP, int(bool(causal)), float(scale), q.ctypes.data, k.ctypes.data, v.ctypes.data,
        int(vstride), pt.ctypes.data, sl.ctypes.data,
        None if rows_arr is None else rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise OracleInputError(_ERRORS.get(rc, f"oracle error {rc}"))
    out, lse = out[:n], lse[:n]
    if rows is None:
        out = out.reshape(B, T, num_q_heads, head_dim_v)
        lse = lse.reshape(B, T, num_q_heads)
    return out, lse


def decode_sparse(*, q, k_pages, v_pages, page_table, seqlens, topk_idx, topk_len, num_q_heads,
                  num_kv_heads, head_dim_qk, head_dim_v, page_size, scale, num_pages=None,
                  v_row_stride=None, rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention of every row over the cache positions its request lists.

    topk_idx: int32 [B][K] (row b lists its positions in entries [0, topk_len[b]));
    topk_len: int32 [B]. Row (b, t, h) attends to the multiset of listed
    positions of request b (a repeat counts twice, no causal mask); see
    ``oracle_decode_sparse_f64``. Other arguments and the return value are
    those of ``decode``.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k_pages, dtype=np.uint16)
    if v_pages is None:
        v = k
        vstride = head_dim_qk if v_row_stride is None else v_row_stride
    else:
        v = np.ascontiguousarray(v_pages, dtype=np.uint16)
        vstride = head_dim_v if v_row_stride is None else v_row_stride
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    ti = np.ascontiguousarray(topk_idx, dtype=np.int32)
    tl = np.ascontiguousarray(topk_len, dtype=np.int32)
    B, T = int(q.shape[0]), int(q.shape[1])
    if ti.ndim != 2 or ti.shape[0] != B or tl.shape != (B,):
        raise OracleInputError("bad shape argument")
    NP = int(k.shape[0]) if num_pages is None else int(num_pages)
    if rows is None:
        n = B * T * num_q_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = int(rows_arr.shape[0])
    out = np.zeros((max(n, 1), head_dim_v), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    rc = lib.oracle_decode_sparse_f64(
        B, T, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, page_size, int(pt.shape[1]), NP,
        float(scale), q.ctypes.data, k.ctypes.data, v.ctypes.data, int(vstride), pt.ctypes.data,
        sl.ctypes.data, ti.ctypes.data, int(max(ti.shape[1], 1)), tl.ctypes.data,
        None if rows_arr is None else rows_arr.ctypes.data, n, out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise OracleInputError(_ERRORS.get(rc, f"oracle error {rc}"))
    out, lse = out[:n], lse[:n]
    if rows is None:
        out = out.reshape(B, T, num_q_heads, head_dim_v)
        lse = lse.reshape(B, T, num_q_heads)
    return out, lse


def decode_workload(w, rows=None):
    """``decode`` on a ``workloads.Workload``."""
    return decode(q=w.q, k_pages=w.k_pages, v_pages=w.v_pages, page_table=w.page_table,
                  seqlens=w.seqlens, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                  head_dim_qk=w.head_dim_qk, head_dim_v=w.head_dim_v, page_size=w.page_size,
                  causal=w.causal, scale=w.scale, v_row_stride=w.v_row_stride, rows=rows)


def decode_sparse_workload(w, rows=None):
    """``decode_sparse`` on a ``workloads.Workload`` that carries a top-k selection."""
    return decode_sparse(q=w.q, k_pages=w.k_pages, v_pages=w.v_pages, page_table=w.page_table,
                         seqlens=w.seqlens, topk_idx=w.topk_idx, topk_len=w.topk_len,
                         num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                         head_dim_qk=w.head_dim_qk, head_dim_v=w.head_dim_v, page_size=w.page_size,
                         scale=w.scale, v_row_stride=w.v_row_stride, rows=rows)


# ---------------------------------------------------------------------------
# split-KV view: partial states and their reduction (fp64, numpy)
# ---------------------------------------------------------------------------

def partial_state(qrow: np.ndarray, keys: np.ndarray, vals: np.ndarray, scale: float):
    """Partial softmax state of one query row over a subset of keys.

    qrow [Dk], keys [n][Dk], vals [n][Dv] (float64). Returns (m, l, acc) with
    m = max_j s_j, l = sum_j exp(s_j - m), acc = sum_j exp(s_j - m) v_j,
    s_j = scale * q.k_j. An empty subset gives (-inf, 0, 0).
    """
    qrow = np.asarray(qrow, np.float64)
    keys = np.asarray(keys, np.float64).reshape(-1, qrow.shape[0])
    vals = np.asarray(vals, np.float64)
    if keys.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(vals.shape[-1])
    s = scale * (keys @ qrow)
    m = float(s.max())
    w = np.exp(s - m)
    return m, float(w.sum()), w @ vals


def merge_states(states):
    """Reduce partial states (m_s, l_s, acc_s) into (out, lse).

    M = max_s m_s; Lambda = sum_s l_s exp(m_s - M);
    out = sum_s acc_s exp(m_s - M) / Lambda; lse = M + ln Lambda.
    All-empty input gives out = 0, lse = -inf.
    """
    ms = np.array([s[0] for s in states], dtype=np.float64)
    M = float(ms.max()) if len(ms) else -np.inf
    dv = len(states[0][2]) if states else 0
    if not np.isfinite(M):
        return np.zeros(dv), -np.inf
    f = np.exp(ms - M)
    lam = float(sum(s[1] * fi for s, fi in zip(states, f)))
    acc = sum(s[2] * fi for s, fi in zip(states, f))
    return acc / lam, M + np.log(lam)


def gather_rows(w, b: int, g: int, n: int):
    """Keys and values (float64) of the first n cache positions of request b, kv head g."""
    from workloads import bf16_bits_to_fp32  # input helper only (no attention arithmetic)
    P = w.page_size
    ks, vs = [], []
    for j in range(n):
        pg = int(w.page_table[b, j // P])
        s = j % P
        ks.append(w.k_pages[pg, s, g if not w.mla else 0])
        if w.mla:
            vs.append(w.k_pages[pg, s, 0, :w.head_dim_v])
        else:
            vs.append(w.v_pages[pg, s, g])
    if n == 0:
        return np.zeros((0, w.head_dim_qk)), np.zeros((0, w.head_dim_v))
    k = bf16_bits_to_fp32(np.stack(ks)).astype(np.float64)
    v = bf16_bits_to_fp32(np.stack(vs)).astype(np.float64)
    return k, v
