// Stream-K split-KV GQA decode attention for sm_103a.
//
// One persistent wave: CTA c walks the segment list the planner gave it (a
// near-equal share of the batch's KV tokens; triton.csdn.net Q&A on waves and
// FlashMLA's Stream-K, closing summary). Per segment (request b, kv-head group
// g, token range) the CTA streams paged K/V with TMA and keeps an online
// softmax per query row ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解",
// section 6.3 / Q8: QK^T -> mask -> softmax -> xV without writing scores to
// HBM). A segment that is only part of its (b, g) item writes its partial
// state (m, l, acc) to an L2-resident workspace slot and counts its arrival;
// the split that arrives last merges the partials right there
// ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", core method:
// just-in-time reduction, no separate reduction kernel and no wait for the
// slowest split). Items with more than 16 splits merge as a two-level tree:
// the last arriver of each run of 16 consecutive splits folds them into one
// partial, and the last of those runs folds the runs. Nobody waits for
// another CTA, so the kernel is correct for any grid size and any scheduling
// order.
//
// CTA layout: warps 0..HG-1 consume (warp h = kv head g*HG + h of the group),
// warp HG (lane 0) produces.
//   stage = one 16-token granule of all HG heads: K and V tiles, each loaded
//           by ONE TMA box of the 5-D map {64 dims, tokens, D/64 halves,
//           heads, pages} (dims listed out of stride order so that the tile
//           lands as [head][half][16 tokens][128 B], 128-byte swizzle: the
//           eight rows an ldmatrix reads are eight different tokens, so the
//           swizzle spreads them over all banks). 32 KB per box for 8 heads
//           of 128 dims: measured on GB300, boxes this large stream at
//           ~7.2 TB/s where 2 KB boxes stall at ~4.9 TB/s.
//   rows  = the G*T query rows of one kv head (padded to 16 for mma.sync
//           m16n8k16; row r is query token r / G, head (kv head)*G + r % G).
#include <math.h>

#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace skd {
namespace {

constexpr int kMaxHG = 8;
constexpr int kMaxStages = 8;
constexpr int kFan = 16;  // splits folded per merge-tree node
constexpr int kTraceWords = SKD_TRACE_RECORD_BYTES / 8;
constexpr int kSmemBudget = 227 * 1024;
constexpr float kLn2 = 0.69314718055994531f;

struct Params {
  const __nv_bfloat16 *q;
  const int32_t *page_table;
  const int32_t *seqlens;
  const int32_t *plan;
  int32_t *err;
  int32_t *item_cnt;   // one per item
  int32_t *group_cnt;  // one per slot (used at the first slot of each run of kFan)
  float *partials;
  __nv_bfloat16 *out;
  float *lse;
  int batch, T, Hq, Hkv, HG, NG, G, P, max_pages, num_pages, causal, rows, max_slots;
  int nst, nq;  // pipeline stages, Q slots
  int stage_bytes, tile_bytes, q_bytes, q_off, zero_off, bar_off, misc_off;
  float scale_log2;
  int64_t slot_floats, head_floats;
  long long *trace;
  int defer;  // 1: splits write their partial states and a combine kernel merges them
};

// Merge `n` partial states of head h (slots base, base+stride, ...) in slot
// order with a running maximum. Final: write out/lse rows; otherwise write the
// folded state into slot `base`. One warp: 8 lanes per row (4 rows at a time),
// each lane owning D/8 consecutive columns; 4-8 splits are loaded per step so
// that a merge costs a few L2 round trips rather than one per split and row.
template <int D>
__device__ void merge_head(const Params &p, int h, int base, int n, int stride, bool final_out,
                           int b, int head, int lane) {
  constexpr int C4 = D / 32;  // float4 per lane per row (D/8 floats)
  constexpr int U = D >= 128 ? 4 : 8;  // splits in flight (register budget: 168/thread)
  const int rows = p.rows;
  const int rg = lane >> 3, cl = lane & 7;
  for (int r0 = 0; r0 < rows; r0 += 4) {
    const int r = r0 + rg;
    const bool act = r < rows;
    float M = -INFINITY, lam = 0.f, lamf = 0.f;
    float4 acc[C4];
#pragma unroll
    for (int c = 0; c < C4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n; s0 += U) {
      float mv[U], lv[U], lfv[U];
      float4 ov[U][C4];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        mv[u] = -INFINITY;
        lv[u] = lfv[u] = 0.f;
#pragma unroll
        for (int c = 0; c < C4; ++c) ov[u][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (act && s0 + u < n) {
          const float *ps = p.partials + int64_t(base + (s0 + u) * stride) * p.slot_floats + h * p.head_floats;
          mv[u] = __ldcg(ps + rows * D + r);
          lv[u] = __ldcg(ps + rows * D + rows + r);
          lfv[u] = __ldcg(ps + rows * D + 2 * rows + r);
          const float4 *o = reinterpret_cast<const float4 *>(ps + r * D + cl * (D / 8));
#pragma unroll
          for (int c = 0; c < C4; ++c) ov[u][c] = __ldcg(o + c);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < U; ++u) Mn = fmaxf(Mn, mv[u]);
      const float Mu = Mn == -INFINITY ? 0.f : Mn;
      const float sc = exp2f(M - Mu);
      lam *= sc;
      lamf *= sc;
#pragma unroll
      for (int c = 0; c < C4; ++c) {
        acc[c].x *= sc;
        acc[c].y *= sc;
        acc[c].z *= sc;
        acc[c].w *= sc;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float f = exp2f(mv[u] - Mu);
        lam += lv[u] * f;
        lamf += lfv[u] * f;
#pragma unroll
        for (int c = 0; c < C4; ++c) {
          acc[c].x += ov[u][c].x * f;
          acc[c].y += ov[u][c].y * f;
          acc[c].z += ov[u][c].z * f;
          acc[c].w += ov[u][c].w * f;
        }
      }
      M = Mn;
    }
    __syncwarp();  // every lane has read slot `base` before it is overwritten
    if (!act) continue;
    if (final_out) {
      const int t = r / p.G;
      const int64_t orow = (int64_t(b) * p.T + t) * p.Hq + int64_t(head) * p.G + (r - t * p.G);
      const float inv = 1.f / lam;
      uint32_t pk[2 * C4];
#pragma unroll
      for (int c = 0; c < C4; ++c) {
        pk[2 * c] = ptx::pack_bf16(acc[c].x * inv, acc[c].y * inv);
        pk[2 * c + 1] = ptx::pack_bf16(acc[c].z * inv, acc[c].w * inv);
      }
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + cl * (D / 8));
#pragma unroll
      for (int c = 0; c < C4 / 2; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (cl == 0) p.lse[orow] = (M + log2f(lamf)) * kLn2;
    } else {
      float *pd = p.partials + int64_t(base) * p.slot_floats + h * p.head_floats;
      float4 *o = reinterpret_cast<float4 *>(pd + r * D + cl * (D / 8));
#pragma unroll
      for (int c = 0; c < C4; ++c) o[c] = acc[c];
      if (cl == 0) {
        pd[rows * D + r] = M;
        pd[rows * D + rows + r] = lam;
        pd[rows * D + 2 * rows + r] = lamf;
      }
    }
  }
}

// The same merge for a CTA's last segment, when its KV ring is idle: whole
// partial-state slots (all HG heads of one split, contiguous) stream through
// the ring as one large bulk copy each, several slots in flight, and every
// consumer warp folds its head's block of each slot in split order with a
// running maximum. One thread of warp 0 issues the copies and refills a buffer
// once all HG warps have released it. `uses` numbers the buffer fills across
// calls (a fold followed by the final merge) so that barrier phases continue.
template <int D>
__device__ __noinline__ bool merge_slots_staged(const Params &p, int h, int HG, int base, int n, int stride,
                                               bool final_out, int b, int head, int lane, uint32_t ring,
                                               uint32_t ring_bytes, const volatile int *abort, int &uses) {
  constexpr int C4 = D / 32;
  const int rows = p.rows;
  const uint32_t sb = uint32_t(p.slot_floats) * 4;
  const int nbuf = min(6, int((ring_bytes - 128) / sb));
  const uint32_t full = ring + ring_bytes - 128, empty = full + 64;
  // lane (rg, cl) handles row 4g + rg and the float4 columns c * 8 + cl, so the
  // eight lanes of a row read 128 contiguous bytes (no bank conflicts)
  const int rg = lane >> 3, cl = lane & 7;
  const int RG = (rows + 3) >> 2;  // row groups of 4 (rows <= 16)
  const bool issuer = h == 0 && lane == 0;
  if (uses == 0 && issuer) {
    for (int k = 0; k < nbuf; ++k) {
      ptx::mbar_init(full + 8 * k, 1);
      ptx::mbar_init(empty + 8 * k, uint32_t(HG));
    }
    ptx::fence_mbar_init();
  }
  // the copies read partial states through the async proxy: order this CTA's
  // own earlier stores to them (a folded run) and the acquired ones of other CTAs
  ptx::fence_proxy_async_global();
  ptx::named_bar(1, HG * 32);
  const int u0 = uses;
  auto fill = [&](int s) {
    const int u = u0 + s, k = u % nbuf;
    ptx::mbar_arrive_expect_tx(full + 8 * k, sb);
    ptx::bulk_load(ring + k * sb, p.partials + int64_t(base + s * stride) * p.slot_floats, sb, full + 8 * k);
  };
  int issued = 0;
  if (issuer)
    for (; issued < min(nbuf, n); ++issued) fill(issued);
  float M[4], lam[4], lamf[4];
  float4 acc[4][C4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    M[k] = -INFINITY;
    lam[k] = lamf[k] = 0.f;
#pragma unroll
    for (int c = 0; c < C4; ++c) acc[k][c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool ok = true;
  for (int s = 0; s < n; ++s) {
    const int u = u0 + s, k = u % nbuf;
    if (ok && !ptx::mbar_wait(full + 8 * k, uint32_t(u / nbuf) & 1u, abort, kWaitCycles)) ok = false;
    const float *bs =
        reinterpret_cast<const float *>(__cvta_shared_to_generic(ring + k * sb)) + int64_t(h) * p.head_floats;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int r = 4 * g + rg;
      if (g < RG && r < rows) {
        const float mv = bs[rows * D + r];
        const float Mn = fmaxf(M[g], mv);
        const float Mu = Mn == -INFINITY ? 0.f : Mn;
        const float sc = exp2f(M[g] - Mu), f = exp2f(mv - Mu);
        lam[g] = lam[g] * sc + bs[rows * D + rows + r] * f;
        lamf[g] = lamf[g] * sc + bs[rows * D + 2 * rows + r] * f;
        const float4 *o = reinterpret_cast<const float4 *>(bs + r * D);
#pragma unroll
        for (int c = 0; c < C4; ++c) {
          const float4 v = o[c * 8 + cl];
          acc[g][c].x = acc[g][c].x * sc + v.x * f;
          acc[g][c].y = acc[g][c].y * sc + v.y * f;
          acc[g][c].z = acc[g][c].z * sc + v.z * f;
          acc[g][c].w = acc[g][c].w * sc + v.w * f;
        }
        M[g] = Mn;
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty + 8 * k);
    if (issuer && ok && issued < n) {
      // the buffer of split s is refilled with split s + nbuf once every warp released it
      if (!ptx::mbar_wait(empty + 8 * k, uint32_t(u / nbuf) & 1u, abort, kWaitCycles)) ok = false;
      if (ok) fill(issued++);
    }
  }
  // after a give-up, the copies still in flight land before the ring is reused
  if (!ok && issuer) {
    atomicOr(p.err, SKD_DEVERR_TIMEOUT);
    for (int s = 0; s < issued; ++s)
      ptx::mbar_wait(full + 8 * ((u0 + s) % nbuf), uint32_t((u0 + s) / nbuf) & 1u, nullptr, kWaitCycles);
  }
  uses = u0 + n;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int r = 4 * g + rg;
    if (g >= RG || r >= rows) continue;
    if (final_out) {
      const int t = r / p.G;
      const int64_t orow = (int64_t(b) * p.T + t) * p.Hq + int64_t(head) * p.G + (r - t * p.G);
      const float inv = 1.f / lam[g];
      uint2 *dst = reinterpret_cast<uint2 *>(p.out + orow * D);
#pragma unroll
      for (int c = 0; c < C4; ++c)
        dst[c * 8 + cl] = make_uint2(ptx::pack_bf16(acc[g][c].x * inv, acc[g][c].y * inv),
                                     ptx::pack_bf16(acc[g][c].z * inv, acc[g][c].w * inv));
      if (cl == 0) p.lse[orow] = (M[g] + log2f(lamf[g])) * kLn2;
    } else {
      float *pd = p.partials + int64_t(base) * p.slot_floats + h * p.head_floats;
      float4 *o = reinterpret_cast<float4 *>(pd + r * D);
#pragma unroll
      for (int c = 0; c < C4; ++c) o[c * 8 + cl] = acc[g][c];
      if (cl == 0) {
        pd[rows * D + r] = M[g];
        pd[rows * D + rows + r] = lam[g];
        pd[rows * D + 2 * rows + r] = lamf[g];
      }
    }
  }
  return ok;
}

template <int D>
__global__ void __launch_bounds__((kMaxHG + 1) * 32, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const Params p) {
  constexpr int NH = D / 64;  // 128-byte halves of a row
  extern __shared__ uint8_t smem_raw[];
  // with programmatic dependent launch this grid may start before the previous
  // kernel of the stream (e.g. the device planner) has finished: wait for it
  // before reading any input
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = p.HG;
  const int32_t *plan = p.plan;

  // A plan built for another launch is rejected by every thread alike.
  if (plan[PH_MAGIC] != kPlanMagic || plan[PH_BATCH] != p.batch || plan[PH_NGRP] != p.NG ||
      plan[PH_NCTAS] != int(gridDim.x) || plan[PH_GRANULE] != kGranule ||
      plan[PH_NSLOTS] > p.max_slots || plan[PH_ERR] != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, plan[PH_ERR] != 0 ? plan[PH_ERR] : SKD_DEVERR_PLAN);
    return;
  }
  const PlanOffsets off = plan_offsets(p.batch, p.NG, gridDim.x);
  const int seg_lo = plan[off.cta_off + blockIdx.x];
  const int seg_hi = plan[off.cta_off + blockIdx.x + 1];
  const int4 *segs = reinterpret_cast<const int4 *>(plan + off.segs);

  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + p.bar_off;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStages + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStages + 2 + s); };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.misc_off);
  volatile int *last_flag = abort_flag + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nst; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), HG);
    }
    for (int s = 0; s < p.nq; ++s) {
      ptx::mbar_init(qfull_bar(s), 1);
      ptx::mbar_init(qempty_bar(s), HG);
    }
    *abort_flag = 0;
    *last_flag = 0;
    ptx::fence_mbar_init();
  }
  // a zero row: A-fragment rows beyond G*T read it
  for (int i = threadIdx.x; i < D * 2 / 16; i += blockDim.x)
    reinterpret_cast<int4 *>(smem + p.zero_off)[i] = make_int4(0, 0, 0, 0);
  __syncthreads();

  const int NG = p.NG, G = p.G, T = p.T, rows = p.rows;
  long long *const tr = p.trace ? p.trace + int64_t(blockIdx.x) * kTraceWords : nullptr;
  if (tr && threadIdx.x == 0) tr[0] = (long long)ptx::globaltimer_ns();
  const long long t_begin = clock64();
  long long t_wait = 0;   // cycles this warp spent in barrier waits (trace only)
  long long t_merge = 0;  // cycles this warp spent publishing and merging partials

  // =========================== producer ====================================
  // The whole warp walks the segments; lane 0 waits on barriers and issues the
  // copies. Page ids of 32 granules are fetched with one coalesced warp load
  // and handed to lane 0 by shuffles.
  if (warp == HG) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
    }
    const uint64_t pol = ptx::policy_evict_first();
    int stage = 0, qs = 0;
    uint32_t phase = 0, qph = 0;
    uint32_t last_parity_mask = 0, used_mask = 0;
    bool ok = true;
    for (int si = seg_lo; si < seg_hi && ok; ++si) {
      const int4 sg = segs[si];
      const int item = sg.x, tb = sg.y, te = sg.z;
      if (te <= tb) continue;
      const int b = item / NG, head0 = (item - b * NG) * HG;
      if (lane == 0) {
        const int L = p.seqlens[b];
        if (te > L || L > p.max_pages * p.P || (p.causal && L < T)) atomicOr(p.err, SKD_DEVERR_SEQLEN);
        const long long w0 = clock64();
        const bool got = ptx::mbar_wait(qempty_bar(qs), qph ^ 1u, abort_flag, kWaitCycles);
        t_wait += clock64() - w0;
        if (!got) {
          ok = false;
        } else {
          const uint32_t per_t = uint32_t(HG * G * D * 2);
          ptx::mbar_arrive_expect_tx(qfull_bar(qs), per_t * T);
          for (int t = 0; t < T; ++t)
            ptx::bulk_load(sbase + p.q_off + qs * p.q_bytes + t * per_t,
                           p.q + ((int64_t(b) * T + t) * p.Hq + int64_t(head0) * G) * D, per_t,
                           qfull_bar(qs));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (++qs == p.nq) {
        qs = 0;
        qph ^= 1u;
      }
      const int32_t *ptab = p.page_table + int64_t(b) * p.max_pages;
      for (int c0 = tb; c0 < te && ok; c0 += 32 * kGranule) {
        const int tk = c0 + lane * kGranule;
        int pg = 0;
        if (tk < te) {
          const int j = tk / p.P;
          pg = j < p.max_pages ? __ldg(ptab + j) : -1;
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.err, SKD_DEVERR_PAGE);
            pg = 0;
          }
        }
        const int cend = min(te, c0 + 32 * kGranule);
        for (int tok0 = c0; tok0 < cend; tok0 += kGranule) {
          const int pgi = __shfl_sync(0xffffffffu, pg, (tok0 - c0) / kGranule);
          if (lane == 0) {
            const long long w0 = clock64();
            const bool got = ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, kWaitCycles);
            t_wait += clock64() - w0;
            if (!got) {
              ok = false;
            } else {
              ptx::mbar_arrive_expect_tx(full_bar(stage), uint32_t(p.stage_bytes));
              const uint32_t kdst = sbase + stage * p.stage_bytes;
              const int slot = tok0 % p.P;
              ptx::tma_load_5d(kdst, &tmK, full_bar(stage), 0, slot, 0, head0, pgi, pol);
              ptx::tma_load_5d(kdst + p.tile_bytes, &tmV, full_bar(stage), 0, slot, 0, head0, pgi, pol);
              used_mask |= 1u << stage;
              last_parity_mask = (last_parity_mask & ~(1u << stage)) | (phase << stage);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (++stage == p.nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, SKD_DEVERR_TIMEOUT);
      }
      // every fill this warp issued must land before the CTA may exit
      for (int s = 0; s < p.nst; ++s)
        if (used_mask & (1u << s))
          ptx::mbar_wait(full_bar(s), (last_parity_mask >> s) & 1u, nullptr, kWaitCycles);
      if (tr) {
        tr[4] = t_wait;
        tr[5] = clock64() - t_begin;
      }
    }
    return;
  }

  // =========================== consumers ===================================
  const int h = warp;            // head within the group
  const int ctid = threadIdx.x;  // 0 .. HG*32-1
  const int cthreads = HG * 32;
  const int fr = lane >> 2, fc = lane & 3;
  const int r0 = fr, r1 = fr + 8;
  const float NEG_INF = -INFINITY;
  int stage = 0, qs = 0;
  uint32_t phase = 0, qph = 0;

  for (int si = seg_lo; si < seg_hi; ++si) {
    const int4 sg = segs[si];
    const int item = sg.x, tb = sg.y, te = sg.z, wslot = sg.w;
    const int b = item / NG;
    const int head = (item - b * NG) * HG + h;
    auto out_row = [&](int r) {
      const int t = r / G;
      return (int64_t(b) * T + t) * p.Hq + int64_t(head) * G + (r - t * G);
    };

    if (te <= tb) {  // empty request: out = 0, lse = -inf
      for (int i = lane; i < rows * (D / 8); i += 32) {
        const int r = i / (D / 8), c = i - r * (D / 8);
        reinterpret_cast<int4 *>(p.out + out_row(r) * D)[c] = make_int4(0, 0, 0, 0);
      }
      for (int r = lane; r < rows; r += 32) p.lse[out_row(r)] = NEG_INF;
      continue;
    }
    const int L = p.seqlens[b];

    // ---- Q fragments (A operand, 16 x D; rows >= G*T read the zero row) ----
    uint32_t qa[D / 16][4];
    bool alive = !*abort_flag;
    {
      const long long w0 = clock64();
      if (alive && !ptx::mbar_wait(qfull_bar(qs), qph, abort_flag, kWaitCycles)) {
        alive = false;
        *abort_flag = 1;
      }
      t_wait += clock64() - w0;
    }
    if (alive) {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      uint32_t rb;
      if (r < rows) {
        const int t = r / G;
        rb = sbase + p.q_off + qs * p.q_bytes + ((t * HG + h) * G + (r - t * G)) * (D * 2);
      } else {
        rb = sbase + p.zero_off;
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ptx::ldsm_x4(rb + (2 * kk + (lane >> 4)) * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      // The Q slot is refilled by TMA as soon as every warp has arrived on
      // qempty, so the fragments must be in registers first: reading them
      // makes in-order issue wait for the loads, and the proxy fence orders
      // these generic reads before the async-proxy writes of the refill.
      uint32_t dep = 0;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) dep |= qa[kk][0] | qa[kk][1] | qa[kk][2] | qa[kk][3];
      asm volatile("" ::"r"(dep));
      ptx::fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(qempty_bar(qs));
    if (++qs == p.nq) {
      qs = 0;
      qph ^= 1u;
    }

    // last visible key of fragment rows r0 and r1 (causal: L - T + t)
    const int lim0 = (p.causal && r0 < rows) ? L - T + r0 / G : INT_MAX;
    const int lim1 = (p.causal && r1 < rows) ? L - T + r1 / G : INT_MAX;

    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    // l: sum of the bf16-rounded p that enter P.V (normalises out, so out is an
    // exact convex combination of V rows); lf: sum of fp32 p (gives lse)
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f, lf0 = 0.f, lf1 = 0.f;

    for (int tok0 = tb; tok0 < te; tok0 += kGranule) {
      {
        const long long w0 = clock64();
        if (alive && !ptx::mbar_wait(full_bar(stage), phase, abort_flag, kWaitCycles)) {
          alive = false;
          *abort_flag = 1;
        }
        t_wait += clock64() - w0;
        if (tr && lane == 0 && h == 0) atomicAdd(reinterpret_cast<unsigned long long *>(tr + 7), 1ull);
      }
      if (alive) {
        const uint32_t kb = sbase + stage * p.stage_bytes + h * (NH * kGranule * 128);
        const uint32_t vb = kb + p.tile_bytes;
        if (tok0 + kGranule > te) {
          // rows past the end of the request hold arbitrary bytes: zero their V
          const int t_lo = te - tok0;
          const int per_half = (kGranule - t_lo) * 8;
          uint8_t *vrow = smem + stage * p.stage_bytes + p.tile_bytes + h * (NH * kGranule * 128);
          for (int c = lane; c < per_half * NH; c += 32) {
            const int hh = c / per_half;
            const int rest = c - hh * per_half;
            const int t = t_lo + (rest >> 3);
            *reinterpret_cast<int4 *>(vrow + (hh * kGranule + t) * 128 + (rest & 7) * 16) =
                make_int4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
        }
        // ---- S = Q K^T over the 16 tokens ----
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int t = (lane & 7) + ((lane >> 4) << 3);
          const int sw = t & 7;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int c = 2 * (kk & 3) + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4(kb + ((kk >> 2) * kGranule + t) * 128 + ((c ^ sw) << 4), b0, b1, b2, b3);
            ptx::mma_bf16_16816(s[0], qa[kk], b0, b1);
            ptx::mma_bf16_16816(s[1], qa[kk], b2, b3);
          }
        }
        // ---- mask, online softmax ----
        float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = tok0 + 8 * j + 2 * fc + e;
            const bool in = tok < te;
            s[j][e] = (in && tok <= lim0) ? s[j][e] * p.scale_log2 : NEG_INF;
            s[j][2 + e] = (in && tok <= lim1) ? s[j][2 + e] * p.scale_log2 : NEG_INF;
            mx0 = fmaxf(mx0, s[j][e]);
            mx1 = fmaxf(mx1, s[j][2 + e]);
          }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == NEG_INF ? 0.f : mn0;
        const float mu1 = mn1 == NEG_INF ? 0.f : mn1;
        const float a0 = exp2f(m0 - mu0), a1 = exp2f(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        uint32_t pa[4];
        float ps0 = 0.f, ps1 = 0.f, pf0 = 0.f, pf1 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float e00 = exp2f(s[j][0] - mu0), e01 = exp2f(s[j][1] - mu0);
          const float e10 = exp2f(s[j][2] - mu1), e11 = exp2f(s[j][3] - mu1);
          pf0 += e00 + e01;
          pf1 += e10 + e11;
          const uint32_t u0 = ptx::pack_bf16(e00, e01);
          const uint32_t u1 = ptx::pack_bf16(e10, e11);
          const float2 f0 = ptx::unpack_bf16(u0), f1 = ptx::unpack_bf16(u1);
          ps0 += f0.x + f0.y;
          ps1 += f1.x + f1.y;
          pa[2 * j] = u0;
          pa[2 * j + 1] = u1;
        }
        l0 = l0 * a0 + ps0;
        l1 = l1 * a1 + ps1;
        lf0 = lf0 * a0 + pf0;
        lf1 = lf1 * a1 + pf1;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          o[j][0] *= a0;
          o[j][1] *= a0;
          o[j][2] *= a1;
          o[j][3] *= a1;
        }
        // ---- O += P V ----
        {
          const int t = (lane & 7) + (((lane >> 3) & 1) << 3);
          const int sw = t & 7;
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj) {
            const int cg = 2 * jj + (lane >> 4);  // 8-column chunk of V
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4_t(vb + ((cg >> 3) * kGranule + t) * 128 + (((cg & 7) ^ sw) << 4), b0, b1, b2,
                           b3);
            ptx::mma_bf16_16816(o[2 * jj], pa, b0, b1);
            ptx::mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty_bar(stage));
      if (++stage == p.nst) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- this warp's head is complete for the segment ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    lf0 += __shfl_xor_sync(0xffffffffu, lf0, 1);
    lf0 += __shfl_xor_sync(0xffffffffu, lf0, 2);
    lf1 += __shfl_xor_sync(0xffffffffu, lf1, 1);
    lf1 += __shfl_xor_sync(0xffffffffu, lf1, 2);
    const bool split = wslot >= 0;
    if (alive) {
      if (!split) {
        const float i0 = 1.f / l0, i1 = 1.f / l1;
        const int64_t o0 = r0 < rows ? out_row(r0) * D : -1, o1 = r1 < rows ? out_row(r1) * D : -1;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          if (o0 >= 0)
            *reinterpret_cast<uint32_t *>(p.out + o0 + 8 * j + 2 * fc) = ptx::pack_bf16(o[j][0] * i0, o[j][1] * i0);
          if (o1 >= 0)
            *reinterpret_cast<uint32_t *>(p.out + o1 + 8 * j + 2 * fc) = ptx::pack_bf16(o[j][2] * i1, o[j][3] * i1);
        }
        if (fc == 0) {
          if (r0 < rows) p.lse[out_row(r0)] = (m0 + log2f(lf0)) * kLn2;
          if (r1 < rows) p.lse[out_row(r1)] = (m1 + log2f(lf1)) * kLn2;
        }
      } else {
        float *ps = p.partials + int64_t(wslot) * p.slot_floats + h * p.head_floats;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          if (r0 < rows) *reinterpret_cast<float2 *>(ps + r0 * D + 8 * j + 2 * fc) = make_float2(o[j][0], o[j][1]);
          if (r1 < rows) *reinterpret_cast<float2 *>(ps + r1 * D + 8 * j + 2 * fc) = make_float2(o[j][2], o[j][3]);
        }
        if (fc == 0) {
          if (r0 < rows) {
            ps[rows * D + r0] = m0;
            ps[rows * D + rows + r0] = l0;
            ps[rows * D + 2 * rows + r0] = lf0;
          }
          if (r1 < rows) {
            ps[rows * D + r1] = m1;
            ps[rows * D + rows + r1] = l1;
            ps[rows * D + 2 * rows + r1] = lf1;
          }
        }
      }
    }
    if (split && !p.defer) {
      // Publish the partial and count arrivals; the last split merges. The
      // barrier orders every consumer thread's partial writes before thread
      // 0's release-acquire atomic, which publishes them GPU-wide.
      const long long tm0 = clock64();
      const int nsp = plan[off.nsplit + item];
      const int s0 = plan[off.slot0 + item];
      const int sidx = wslot - s0;
      const int k = sidx / kFan;
      ptx::named_bar(1, cthreads);
      if (ctid == 0) {
        int last = 0;
        if (!*abort_flag) {
          if (nsp <= kFan) {
            last = ptx::atom_add_acq_rel_gpu(p.item_cnt + item, 1) == nsp - 1 ? 2 : 0;
          } else {
            const int gsz = min(kFan, nsp - k * kFan);
            last = ptx::atom_add_acq_rel_gpu(p.group_cnt + s0 + k * kFan, 1) == gsz - 1 ? 1 : 0;
          }
        }
        *last_flag = last;
      }
      ptx::named_bar(1, cthreads);
      int last = *last_flag;
      // merges of many splits in this CTA's last segment go through its idle KV ring
      const uint32_t ring_bytes = uint32_t(p.nst * p.stage_bytes);
      const bool can_stage = si == seg_hi - 1 && ring_bytes >= 2 * uint32_t(p.slot_floats) * 4 + 128;
      int staged_uses = 0;
      auto merge = [&](int mbase, int mn, int mstride, bool fin) {
        if (can_stage && mn >= 8)
          merge_slots_staged<D>(p, h, HG, mbase, mn, mstride, fin, b, head, lane, sbase, ring_bytes, abort_flag,
                                staged_uses);
        else
          merge_head<D>(p, h, mbase, mn, mstride, fin, b, head, lane);
      };
      if (last == 1) {  // fold this run of kFan splits into its first slot
        const int gsz = min(kFan, nsp - k * kFan);
        merge(s0 + k * kFan, gsz, 1, false);
        ptx::named_bar(1, cthreads);
        if (ctid == 0) {
          if (tr) atomicAdd(reinterpret_cast<unsigned long long *>(tr + 11), 1ull);
          p.group_cnt[s0 + k * kFan] = 0;
          const int ngroups = (nsp + kFan - 1) / kFan;
          *last_flag = ptx::atom_add_acq_rel_gpu(p.item_cnt + item, 1) == ngroups - 1 ? 3 : 0;
        }
        ptx::named_bar(1, cthreads);
        last = *last_flag;
      }
      if (last >= 2) {  // final merge: all splits (2) or all runs (3)
        if (last == 2)
          merge(s0, nsp, 1, true);
        else
          merge(s0, (nsp + kFan - 1) / kFan, kFan, true);
        if (ctid == 0) {
          p.item_cnt[item] = 0;
          if (tr) atomicAdd(reinterpret_cast<unsigned long long *>(tr + 10), 1ull);
        }
      }
      t_merge += clock64() - tm0;
    }
    ptx::named_bar(1, cthreads);  // last_flag is reused by the next segment
  }
  if (tr && lane == 0) {
    atomicAdd(reinterpret_cast<unsigned long long *>(tr + 2), (unsigned long long)t_wait);
    atomicAdd(reinterpret_cast<unsigned long long *>(tr + 3), (unsigned long long)(clock64() - t_begin));
    atomicAdd(reinterpret_cast<unsigned long long *>(tr + 9), (unsigned long long)t_merge);
    if (h == 0) {
      tr[6] = seg_hi - seg_lo;
      tr[8] = ptx::smid();
      tr[1] = (long long)ptx::globaltimer_ns();
    }
  }
}

// The comparator's second kernel: one CTA per work item, warp h merges head h
// of the item's splits (all of them, in split order) and writes out / lse.
template <int D>
__global__ void __launch_bounds__(kMaxHG * 32, 1) gqa_combine_kernel(const Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int item = blockIdx.x, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PlanOffsets off = plan_offsets(p.batch, p.NG, p.plan[PH_NCTAS]);
  const int nsp = p.plan[off.nsplit + item], s0 = p.plan[off.slot0 + item];
  if (nsp < 2 || h >= p.HG) return;
  const int b = item / p.NG, head = (item - b * p.NG) * p.HG + h;
  merge_head<D>(p, h, s0, nsp, 1, true, b, head, lane);
}

template <int D>
int launch_combine_d(const DecodeArgs &a) {
  const skd_shape_t &s = a.shape;
  const int HG = head_group(s.num_kv_heads);
  Params p = {};
  p.plan = a.plan;
  uint8_t *ws = static_cast<uint8_t *>(a.ws);
  p.partials = reinterpret_cast<float *>(ws + a.wl.partials);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.batch = s.batch;
  p.T = s.q_tokens;
  p.Hq = s.num_q_heads;
  p.HG = HG;
  p.NG = s.num_kv_heads / HG;
  p.G = s.num_q_heads / s.num_kv_heads;
  p.rows = p.G * s.q_tokens;
  p.slot_floats = a.wl.slot_floats;
  p.head_floats = a.wl.head_floats;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.batch * p.NG);
  cfg.blockDim = dim3(HG * 32);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gqa_combine_kernel<D>, p) != cudaSuccess) return SKD_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

template <int D>
int launch_d(const DecodeArgs &a) {
  constexpr int NH = D / 64;
  const skd_shape_t &s = a.shape;
  const int HG = head_group(s.num_kv_heads);
  const int G = s.num_q_heads / s.num_kv_heads;
  CUtensorMap tk, tv;
  // dims (innermost first): 64 dims, page slot, 128-byte half, kv head, page
  const cuuint64_t gd[5] = {64, cuuint64_t(s.page_size), cuuint64_t(NH), cuuint64_t(s.num_kv_heads),
                            cuuint64_t(s.num_pages)};
  const cuuint64_t sk[4] = {cuuint64_t(s.num_kv_heads) * D * 2, 128, cuuint64_t(D) * 2,
                            cuuint64_t(s.page_size) * s.num_kv_heads * D * 2};
  const cuuint64_t sv[4] = {cuuint64_t(s.num_kv_heads) * s.v_row_stride * 2, 128,
                            cuuint64_t(s.v_row_stride) * 2,
                            cuuint64_t(s.page_size) * s.num_kv_heads * s.v_row_stride * 2};
  const cuuint32_t box[5] = {64, cuuint32_t(kGranule), cuuint32_t(NH), cuuint32_t(HG), 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  if (encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(a.k), gd, sk, box, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return SKD_EINVAL;
  if (encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(a.v), gd, sv, box, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return SKD_EINVAL;

  Params p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.page_table = a.page_table;
  p.seqlens = a.seqlens;
  p.plan = a.plan;
  uint8_t *ws = static_cast<uint8_t *>(a.ws);
  p.err = reinterpret_cast<int32_t *>(ws);
  p.item_cnt = reinterpret_cast<int32_t *>(ws + a.wl.counters);
  p.group_cnt = reinterpret_cast<int32_t *>(ws + a.wl.group_counters);
  p.partials = reinterpret_cast<float *>(ws + a.wl.partials);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.batch = s.batch;
  p.T = s.q_tokens;
  p.Hq = s.num_q_heads;
  p.Hkv = s.num_kv_heads;
  p.HG = HG;
  p.NG = s.num_kv_heads / HG;
  p.G = G;
  p.P = s.page_size;
  p.max_pages = s.max_pages_per_req;
  p.num_pages = s.num_pages;
  p.causal = s.causal ? 1 : 0;
  p.rows = G * s.q_tokens;
  p.max_slots = int(a.wl.slots);
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.slot_floats = a.wl.slot_floats;
  p.head_floats = a.wl.head_floats;
  p.trace = static_cast<long long *>(trace_buffer(a.n_ctas));
  p.defer = a.defer_merge ? 1 : 0;

  // shared memory: stages | Q slots | zero row | barriers | flags
  p.tile_bytes = HG * NH * kGranule * 128;
  p.stage_bytes = 2 * p.tile_bytes;
  p.q_bytes = ((HG * G * s.q_tokens * D * 2) + 127) / 128 * 128;
  const int fixed = D * 2 + (2 * kMaxStages + 4) * 8 + 16 + 1024;
  p.nq = 2;
  p.nst = std::min(kMaxStages, (kSmemBudget - fixed - 2 * p.q_bytes) / p.stage_bytes);
  if (p.nst < 3) {
    p.nq = 1;
    p.nst = std::min(kMaxStages, (kSmemBudget - fixed - p.q_bytes) / p.stage_bytes);
  }
  if (p.nst < 2) return SKD_EUNSUPPORTED;
  p.q_off = p.nst * p.stage_bytes;
  p.zero_off = p.q_off + p.nq * p.q_bytes;
  p.bar_off = p.zero_off + D * 2;
  p.misc_off = p.bar_off + (2 * kMaxStages + 4) * 8;
  const int smem = p.misc_off + 16 + 1024;

  static bool attr_set = false;  // per process; the attribute belongs to the function
  if (!attr_set) {
    if (cudaFuncSetAttribute(gqa_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBudget) != cudaSuccess)
      return SKD_ECUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_ctas);
  cfg.blockDim = dim3((HG + 1) * 32);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gqa_decode_kernel<D>, tk, tv, p) != cudaSuccess) return SKD_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace

int launch_gqa_combine(const DecodeArgs &a) {
  if (a.shape.batch == 0) return SKD_OK;
  if (a.shape.head_dim_qk == 128) return launch_combine_d<128>(a);
  if (a.shape.head_dim_qk == 64) return launch_combine_d<64>(a);
  return SKD_EUNSUPPORTED;
}

int launch_gqa(const DecodeArgs &a) {
  const int D = a.shape.head_dim_qk;
  if (a.shape.head_dim_v != D) return SKD_EUNSUPPORTED;
  if ((a.shape.num_q_heads / a.shape.num_kv_heads) * a.shape.q_tokens > 16) return SKD_EUNSUPPORTED;
  if (D == 128) return launch_d<128>(a);
  if (D == 64) return launch_d<64>(a);
  return SKD_EUNSUPPORTED;
}

}  // namespace skd

// ---------------------------------------------------------------------------
// Allocation-free entry point. Some callers cannot allocate device memory for
// a workspace: operator plugins whose fixed interface has no scratch argument,
// or runtimes whose memory is planned up front by a framework allocator that
// forbids further cudaMalloc calls. For them the workspace (error word,
// arrival counters, partial softmax states) lives in a fixed module-scope
// device array of kNoAllocScratchBytes, which every GPU that loads this library
// holds until the process exits.
namespace skd {
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];  // device address of the array, per device
}  // namespace

}  // namespace skd

extern "C" int skd_decode_attention_noalloc(const skd_shape_t *shape, const void *q,
                                            const void *k_pages, const void *v_pages,
                                            const int32_t *page_table, const int32_t *seqlens,
                                            const void *plan_dev, int n_ctas, void *out,
                                            float *lse, void *stream) {
  using namespace skd;
  if (!shape || shape->kind != SKD_KIND_GQA) return shape ? SKD_EUNSUPPORTED : SKD_EINVAL;
  const size_t need = skd_workspace_bytes(shape, n_ctas);
  if (need == 0) return n_ctas < 1 ? SKD_EINVAL : SKD_EUNSUPPORTED;
  if (need > kNoAllocScratchBytes) return SKD_ESIZE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SKD_ECUDA;
  void *ws = nullptr;
  {
    // first call on this device: look up the array's device address (host code
    // only sees a host-side stand-in for the symbol)
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SKD_ECUDA;
      g_noalloc_ptr[dev] = ptr;
    }
    ws = g_noalloc_ptr[dev];
  }
  // the error word and the counters must start at zero; the partial slots are
  // always written before they are read
  const WsLayout wl = ws_layout(*shape, n_ctas);
  if (cudaMemsetAsync(ws, 0, size_t(wl.partials), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SKD_ECUDA;
  return skd_decode_attention(shape, q, k_pages, v_pages, page_table, seqlens, plan_dev, n_ctas, ws,
                              kNoAllocScratchBytes, out, lse, stream);
}

