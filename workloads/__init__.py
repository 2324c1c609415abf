"""Seeded synthetic decode-attention workloads.

This module only draws inputs. It holds none of the attention arithmetic, so the
CUDA path and the fp64 oracle can both consume what it produces without sharing
any code with each other.

Recipe (fixed order of draws from one numpy PCG64 stream per workload):
  1. seqlens            (integers, distribution per workload)
  2. physical page ids   (a random permutation of all pages the batch needs)
  3. q                   bf16 ~ N(0, 1), layout [B][T][Hq][Dk]
  4. k_pages             bf16 ~ N(0, 1), layout [NP][P][Hkv][Dk]
  5. v_pages             bf16 ~ N(0, 1), layout [NP][P][Hkv][Dv]   (GQA only)
For the absorbed-MLA workload there is one latent cache [NP][P][576]; V is the
first 512 columns of the same rows (row stride 576), so step 5 is skipped.

A top-k selection (sparse MLA) is drawn afterwards from its own stream
(PCG64 seeded with [seed, 1]), so the cache draws above do not change: request b
lists K_b = min(k, L_b) distinct positions of [0, L_b), sampled uniformly, in
random order (an indexer's top-k comes ordered by score, not by position).

bf16 values are produced by rounding fp32 normals to nearest-even; they are kept
as uint16 bit patterns so that nothing here depends on a bf16 dtype.
Page-table entries past a request's last page are -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "make",
    "make_custom",
    "select_topk",
    "share_prefix",
    "fp32_to_bf16_bits",
    "bf16_bits_to_fp32",
]


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, n: int, chunk: int = 1 << 20) -> np.ndarray:
    """n fp32 N(0,1) draws rounded to bf16 (same values as fp32_to_bf16_bits of
    one big draw; chunked only to avoid large temporaries)."""
    out = np.empty(n, dtype=np.uint16)
    buf = np.empty(chunk, dtype=np.float32)
    u = buf.view(np.uint32)
    tmp = np.empty(chunk, dtype=np.uint32)
    for s in range(0, n, chunk):
        m = min(n, s + chunk) - s
        rng.standard_normal(out=buf[:m], dtype=np.float32)
        t = tmp[:m]
        np.right_shift(u[:m], 16, out=t)
        np.bitwise_and(t, 1, out=t)
        np.add(t, 0x7FFF, out=t)
        np.add(u[:m], t, out=t)
        np.right_shift(t, 16, out=t)
        out[s:s + m] = t
    return out


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    q_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    page_size: int
    causal: bool
    scale: float
    mla: bool
    seqlens: np.ndarray          # int32 [B]
    page_table: np.ndarray       # int32 [B][max_pages]
    q: np.ndarray                # uint16 (bf16 bits) [B][T][Hq][Dk]
    k_pages: np.ndarray          # uint16 [NP][P][Hkv][Dk]
    v_pages: Optional[np.ndarray]  # uint16 [NP][P][Hkv][Dv]; None for MLA (V aliases k_pages)
    seed: int = 0
    topk_idx: Optional[np.ndarray] = None  # int32 [B][K]: listed cache positions (sparse attention)
    topk_len: Optional[np.ndarray] = None  # int32 [B]: entries of row b that are listed
    prefix_groups: Optional[list] = None   # lists of requests whose first pages are shared
    prefix_lens: Optional[list] = None     # shared prefix length (tokens) of each group

    @property
    def sparse(self) -> bool:
        return self.topk_idx is not None

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def v_row_stride(self) -> int:
        """Elements between consecutive V rows ((page, slot, head) triples)."""
        return self.head_dim_qk if self.mla else self.head_dim_v

    @property
    def kv_tokens(self) -> int:
        """KV rows the attention reads: all cached tokens, or the listed ones;
        with shared prefixes, each group's prefix once."""
        if self.sparse:
            return int(self.topk_len.astype(np.int64).sum())
        n = int(self.seqlens.astype(np.int64).sum())
        if self.prefix_groups:
            n -= sum((len(g) - 1) * int(lp) for g, lp in zip(self.prefix_groups, self.prefix_lens))
        return n

    def kv_bytes_per_token(self) -> int:
        if self.mla:
            return self.head_dim_qk * 2
        return self.num_kv_heads * (self.head_dim_qk + self.head_dim_v) * 2

    def algorithmic_bytes(self) -> int:
        """KV bytes + q + out (bf16) + lse (fp32) + referenced page-table entries
        (sparse: one page-table entry and one index per listed position)."""
        P = self.page_size
        if self.sparse:
            pages = 2 * self.kv_tokens
        else:
            pages = int(sum((int(L) + P - 1) // P for L in self.seqlens))
            if self.prefix_groups:
                pages -= sum((len(g) - 1) * int(lp) // P for g, lp in zip(self.prefix_groups, self.prefix_lens))
        rows = self.batch * self.q_tokens * self.num_q_heads
        return (self.kv_tokens * self.kv_bytes_per_token()
                + rows * self.head_dim_qk * 2 + rows * self.head_dim_v * 2 + rows * 4 + pages * 4)

    def algorithmic_flops(self) -> int:
        """2 * T * Hq * (Dk + Dv) per visible KV token (causal rows see fewer)."""
        tot = 0
        for L in self.seqlens:
            L = int(L)
            for t in range(self.q_tokens):
                n = (L - self.q_tokens + t + 1) if (self.causal and L > 0) else L
                tot += 2 * self.num_q_heads * (self.head_dim_qk + self.head_dim_v) * max(n, 0)
        return tot

    def describe(self) -> dict:
        return dict(workload=self.name, batch=self.batch, q_tokens=self.q_tokens,
                    num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
                    head_dim_qk=self.head_dim_qk, head_dim_v=self.head_dim_v,
                    page_size=self.page_size, causal=self.causal, mla=self.mla,
                    kv_tokens=self.kv_tokens, seed=self.seed,
                    **({"topk": int(self.topk_idx.shape[1])} if self.sparse else {}),
                    **({"prefix_groups": [len(g) for g in self.prefix_groups],
                        "prefix_lens": [int(x) for x in self.prefix_lens]} if self.prefix_groups else {}))


def _assemble(name, rng, seqlens, *, T, Hq, Hkv, Dk, Dv, P, causal, scale, mla, seed,
              max_pages=None, spare_pages=0) -> Workload:
    seqlens = np.asarray(seqlens, dtype=np.int32)
    B = int(seqlens.shape[0])
    need = [(int(L) + P - 1) // P for L in seqlens]
    NP = int(sum(need)) + int(spare_pages)
    mp = max(1, max(need) if need else 1) if max_pages is None else int(max_pages)
    perm = rng.permutation(max(NP, 1)).astype(np.int32)[:NP]
    table = np.full((B, mp), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[o:o + n]
        o += n
    q = _normal_bf16(rng, B * T * Hq * Dk).reshape(B, T, Hq, Dk)
    npg = max(NP, 1)
    if mla:
        k = _normal_bf16(rng, npg * P * Dk).reshape(npg, P, 1, Dk)
        v = None
    else:
        k = _normal_bf16(rng, npg * P * Hkv * Dk).reshape(npg, P, Hkv, Dk)
        v = _normal_bf16(rng, npg * P * Hkv * Dv).reshape(npg, P, Hkv, Dv)
    return Workload(name=name, batch=B, q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim_qk=Dk, head_dim_v=Dv, page_size=P, causal=causal, scale=scale,
                    mla=mla, seqlens=seqlens, page_table=table, q=q, k_pages=k, v_pages=v,
                    seed=seed)


def _tiny_gqa(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return _assemble("tiny_gqa_b2_h8kv2_d64", rng, [37, 200], T=1, Hq=8, Hkv=2, Dk=64, Dv=64,
                     P=16, causal=False, scale=1.0 / math.sqrt(64), mla=False, seed=seed)


def _llama3_8b(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    L = rng.integers(512, 8192, size=32, endpoint=True)
    return _assemble("llama3_8b_gqa_b32_h32kv8_d128_p16", rng, L, T=1, Hq=32, Hkv=8, Dk=128,
                     Dv=128, P=16, causal=False, scale=1.0 / math.sqrt(128), mla=False, seed=seed)


def _skewed(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    short = rng.integers(64, 1024, size=63, endpoint=True)
    pos = int(rng.integers(0, 64))
    L = np.insert(short, pos, 131072)
    return _assemble("skewed_gqa_b64_h64kv8_d128_p64_1x131072", rng, L, T=1, Hq=64, Hkv=8,
                     Dk=128, Dv=128, P=64, causal=False, scale=1.0 / math.sqrt(128), mla=False,
                     seed=seed)


def _mla(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    L = rng.integers(1024, 16384, size=64, endpoint=True)
    return _assemble("mla_absorbed_b64_h128_d576v512_p64", rng, L, T=1, Hq=128, Hkv=1, Dk=576,
                     Dv=512, P=64, causal=False, scale=1.0 / math.sqrt(576), mla=True, seed=seed)


def select_topk(w: Workload, k: int, seed: Optional[int] = None, name: Optional[str] = None) -> Workload:
    """The same cache with a top-k selection per request (see the module docstring)."""
    rng = np.random.Generator(np.random.PCG64([w.seed if seed is None else seed, 1]))
    B = w.batch
    idx = np.zeros((B, max(k, 1)), dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        L = int(w.seqlens[b])
        kb = min(k, L)
        if kb > 0:
            idx[b, :kb] = rng.permutation(rng.choice(L, size=kb, replace=False)).astype(np.int32)
        n[b] = kb
    return dataclasses.replace(w, topk_idx=idx, topk_len=n, name=name or w.name + f"_top{k}")


def share_prefix(w: Workload, groups, prefix_lens, name: Optional[str] = None) -> Workload:
    """The same batch where each group's requests share their first
    prefix_len tokens: every member's page table lists the first member's
    pages for them (the members' own prefix pages are left unused)."""
    pt = w.page_table.copy()
    for g, lp in zip(groups, prefix_lens):
        npg = int(lp) // w.page_size
        assert int(lp) % w.page_size == 0 and all(int(w.seqlens[b]) >= int(lp) for b in g)
        for b in g[1:]:
            pt[b, :npg] = pt[g[0], :npg]
    return dataclasses.replace(w, page_table=pt, prefix_groups=[list(g) for g in groups],
                               prefix_lens=[int(x) for x in prefix_lens], name=name or w.name + "_shared")


def _shared_prefix(seed):
    """Llama-3-8B-shaped GQA decode, 8 groups of 4 requests sharing a
    4096-token prefix (a system prompt / few-shot context), own suffixes
    U[64, 1024]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    suffix = rng.integers(64, 1024, size=32, endpoint=True)
    w = _assemble("shared_prefix_gqa", rng, 4096 + suffix, T=1, Hq=32, Hkv=8, Dk=128, Dv=128, P=16,
                  causal=False, scale=1.0 / math.sqrt(128), mla=False, seed=seed)
    groups = [list(range(4 * i, 4 * i + 4)) for i in range(8)]
    return share_prefix(w, groups, [4096] * 8, name="shared_prefix_gqa_b32_8x4_p4096_h32kv8_d128_p16")


def _mla_sparse(seed):
    return select_topk(_mla(seed), 2048, name="mla_sparse_top2048_b64_h128_d576v512_p64")


def _speculative(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    L = rng.integers(4096, 32768, size=16, endpoint=True)
    return _assemble("speculative_gqa_b16_t4_h32kv8_d128_p16", rng, L, T=4, Hq=32, Hkv=8,
                     Dk=128, Dv=128, P=16, causal=True, scale=1.0 / math.sqrt(128), mla=False,
                     seed=seed)


WORKLOADS = {
    "tiny_gqa": _tiny_gqa,
    "llama3_8b_gqa": _llama3_8b,
    "skewed_gqa": _skewed,
    "mla_absorbed": _mla,
    "speculative_gqa": _speculative,
    "mla_sparse_top2048": _mla_sparse,
    "shared_prefix_gqa": _shared_prefix,
}


def make(name: str, seed: int = 0) -> Workload:
    """Build one of the named workloads (full size)."""
    return WORKLOADS[name](seed)


def make_custom(seqlens: Sequence[int], *, q_tokens=1, num_q_heads=8, num_kv_heads=2,
                head_dim_qk=64, head_dim_v=None, page_size=16, causal=None, scale=None,
                mla=False, seed=0, max_pages=None, spare_pages=0, name="custom") -> Workload:
    """Small seeded workloads for tests (same draw order as the named ones)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    Dv = head_dim_qk if head_dim_v is None else head_dim_v
    if mla:
        num_kv_heads = 1
    if causal is None:
        causal = q_tokens > 1
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim_qk)
    return _assemble(name, rng, list(seqlens), T=q_tokens, Hq=num_q_heads, Hkv=num_kv_heads,
                     Dk=head_dim_qk, Dv=Dv, P=page_size, causal=bool(causal), scale=float(scale),
                     mla=mla, seed=seed, max_pages=max_pages, spare_pages=spare_pages)


def draw_seqlens(name: str, seed: int = 0) -> np.ndarray:
    """Only the seqlens of a named workload (first draw of its stream)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny_gqa":
        return np.array([37, 200], dtype=np.int32)
    if name == "llama3_8b_gqa":
        return rng.integers(512, 8192, size=32, endpoint=True).astype(np.int32)
    if name == "skewed_gqa":
        short = rng.integers(64, 1024, size=63, endpoint=True)
        pos = int(rng.integers(0, 64))
        return np.insert(short, pos, 131072).astype(np.int32)
    if name in ("mla_absorbed", "mla_sparse_top2048"):
        return rng.integers(1024, 16384, size=64, endpoint=True).astype(np.int32)
    if name == "shared_prefix_gqa":
        return (4096 + rng.integers(64, 1024, size=32, endpoint=True)).astype(np.int32)
    if name == "speculative_gqa":
        return rng.integers(4096, 32768, size=16, endpoint=True).astype(np.int32)
    raise KeyError(name)
