// Device planner: the Stream-K one-wave split computed by one CTA from device
// seqlens, so that planning and attention can be captured together in a CUDA
// graph ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 7: a graph
// replays fixed launches; here the plan buffer has a fixed size).
//
// It produces the same bytes as the host planner (triton.csdn.net Q&A on
// waves and FlashMLA's Stream-K, closing summary: cut the total work into as
// many near-equal chunks as there are SMs). The host planner sweeps
// sequentially; this kernel computes each item's CTA range in closed form:
// with bound(c) = floor(c*total/n), the CTA containing granule x is
// ceil((x+1)*n/total) - 1, and the segments of a CTA are a contiguous range of
// item indices, so an item's slot in its CTA's list is (item - first item).
#include "kernels.h"
#include "plan_layout.h"

namespace skd {
namespace {

constexpr int kPlanThreads = 1024;

// CTA owning granule position x (x == total -> last CTA)
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t total, int64_t n) {
  if (total == 0 || x >= total) return n - 1;
  const int64_t c = ((x + 1) * n + total - 1) / total - 1;
  return c < n - 1 ? c : n - 1;
}

// Walks bound(c) = floor(c*total/n) for c = c0, c0+1, ... with one division at
// the start and additions after it (an item can span hundreds of CTAs, and a
// 64-bit division per step made the planner slow for short batches).
struct BoundWalk {
  int64_t lo, hi, q, r, acc, n;  // lo = bound(c), hi = bound(c+1), acc = (c+1)*total mod n
  __device__ BoundWalk(int64_t c, int64_t total, int64_t n_) : n(n_) {
    q = total / n;
    r = total - q * n;
    lo = (c * total) / n;
    const int64_t x = (c + 1) * total;
    hi = x / n;
    acc = x - hi * n;
  }
  __device__ void next() {
    lo = hi;
    hi += q;
    acc += r;
    if (acc >= n) {
      acc -= n;
      ++hi;
    }
  }
};

// In-place exclusive scan of a[0..len) (int32) by the whole block; returns the total.
__device__ int block_exclusive_scan(int32_t *a, int len, int32_t *warp_sums, int32_t *carry_sm) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) *carry_sm = 0;
  __syncthreads();
  for (int base = 0; base < len; base += kPlanThreads) {
    const int i = base + tid;
    int v = i < len ? a[i] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int ws = warp_sums[lane];
      int z = ws;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      warp_sums[lane] = z - ws;  // exclusive
      if (lane == 31) warp_sums[32] = z;
    }
    __syncthreads();
    const int carry = *carry_sm;
    if (i < len) a[i] = carry + warp_sums[wid] + x - v;
    __syncthreads();
    if (tid == 0) *carry_sm = carry + warp_sums[32];
    __syncthreads();
  }
  return *carry_sm;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_device_kernel(const int32_t *__restrict__ seqlens, int batch, int ngrp, int n, int seg_cost, int align,
                       int32_t *__restrict__ plan) {
  extern __shared__ int32_t sm[];
  int32_t *req_pref = sm;                 // [batch + 1] virtual-unit prefix per request
  int32_t *cnt = req_pref + batch + 1;    // [n + 1] segments per CTA -> offsets
  int32_t *first = cnt + n + 1;           // [n] smallest item of each CTA
  __shared__ int32_t warp_sums[33];
  __shared__ int32_t carry;
  __shared__ int32_t err;
  const int tid = threadIdx.x;
  const int unit = kGranule * align;                 // tokens per cut unit
  const int vcost = (seg_cost + align - 1) / align;  // virtual units per item
  // the attention kernel that follows may be scheduled now: it waits for this
  // grid to complete (griddepcontrol.wait) before reading the plan
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const PlanOffsets off = plan_offsets(batch, ngrp, n);
  const int64_t items = int64_t(batch) * ngrp;
  int32_t *nsplit = plan + off.nsplit;
  int32_t *slot0 = plan + off.slot0;
  int4 *segs = reinterpret_cast<int4 *>(plan + off.segs);

  if (tid == 0) err = 0;
  __syncthreads();
  for (int b = tid; b < batch; b += kPlanThreads) {
    const int L = seqlens[b];
    if (L < 0) atomicOr(&err, SKD_DEVERR_SEQLEN);
    // each of the request's ngrp items: its segment cost, then its units
    req_pref[b] = L > 0 ? (L + unit - 1) / unit + vcost : 0;
  }
  for (int c = tid; c <= n; c += kPlanThreads) cnt[c] = 0;
  for (int c = tid; c < n; c += kPlanThreads) first[c] = 0x7fffffff;
  __syncthreads();
  const int32_t req_total = block_exclusive_scan(req_pref, batch, warp_sums, &carry);
  if (tid == 0) req_pref[batch] = req_total;
  __syncthreads();
  const int64_t total = int64_t(ngrp) * req_pref[batch];
  if (tid == 0 && total > 0x7fffffffLL) err |= SKD_DEVERR_SEQLEN;
  __syncthreads();
  if (err) {
    // a plan that every kernel rejects: header with the error bits set
    for (int64_t i = tid; i < off.words; i += kPlanThreads) plan[i] = 0;
    __syncthreads();
    if (tid == 0) {
      plan[PH_MAGIC] = kPlanMagic;
      plan[PH_BATCH] = batch;
      plan[PH_NGRP] = ngrp;
      plan[PH_NCTAS] = n;
      plan[PH_GRANULE] = kGranule;
      plan[PH_ERR] = err;
    }
    return;
  }

  // pass 1: per item, the CTAs it touches; count segments per CTA
  for (int64_t i = tid; i < items; i += kPlanThreads) {
    const int b = int(i / ngrp), h = int(i - int64_t(b) * ngrp);
    const int64_t gv = req_pref[b + 1] - req_pref[b];  // virtual length of each item of b
    const int64_t g = gv > 0 ? gv - vcost : 0;
    const int64_t s = int64_t(ngrp) * req_pref[b] + h * gv + (gv - g), e = s + g;
    int ns = 0;
    if (g == 0) {
      const int64_t c = cta_of(s, total, n);
      atomicAdd(&cnt[c], 1);
      atomicMin(&first[c], int(i));
      ns = 1;
    } else {
      const int64_t cf = cta_of(s, total, n), cl = cta_of(e - 1, total, n);
      BoundWalk bw(cf, total, n);
      for (int64_t c = cf; c <= cl; ++c, bw.next()) {
        if (bw.hi <= bw.lo) continue;  // empty chunk
        atomicAdd(&cnt[c], 1);
        atomicMin(&first[c], int(i));
        ++ns;
      }
    }
    nsplit[i] = ns;
  }
  __syncthreads();
  const int nseg = block_exclusive_scan(cnt, n, warp_sums, &carry);
  if (tid == 0) cnt[n] = nseg;
  __syncthreads();
  for (int c = tid; c <= n; c += kPlanThreads) plan[off.cta_off + c] = cnt[c];
  // slots: consecutive per item with more than one split, in item order
  for (int64_t i = tid; i < items; i += kPlanThreads) slot0[i] = nsplit[i] > 1 ? nsplit[i] : 0;
  __syncthreads();
  const int nslots = block_exclusive_scan(slot0, int(items), warp_sums, &carry);
  __syncthreads();
  // pass 2: write segments
  for (int64_t i = tid; i < items; i += kPlanThreads) {
    const int b = int(i / ngrp), h = int(i - int64_t(b) * ngrp);
    const int L = seqlens[b];
    const int64_t gv = req_pref[b + 1] - req_pref[b];
    const int64_t g = gv > 0 ? gv - vcost : 0;
    const int64_t s = int64_t(ngrp) * req_pref[b] + h * gv + (gv - g), e = s + g;
    const int ns = nsplit[i];
    const int sl0 = ns > 1 ? slot0[i] : -1;
    if (g == 0) {
      const int64_t c = cta_of(s, total, n);
      segs[cnt[c] + (i - first[c])] = make_int4(int(i), 0, 0, -1);
    } else {
      const int64_t cf = cta_of(s, total, n), cl = cta_of(e - 1, total, n);
      int k = 0;
      BoundWalk bw(cf, total, n);
      for (int64_t c = cf; c <= cl; ++c, bw.next()) {
        const int64_t lo_c = bw.lo, hi_c = bw.hi;
        if (hi_c <= lo_c) continue;
        const int64_t lo = s > lo_c ? s : lo_c, hi = e < hi_c ? e : hi_c;
        const int64_t tb = (lo - s) * unit;
        const int64_t te = (hi - s) * unit < L ? (hi - s) * unit : L;
        segs[cnt[c] + (i - first[c])] = make_int4(int(i), int(tb), int(te), ns > 1 ? sl0 + k : -1);
        ++k;
      }
    }
    slot0[i] = sl0;
  }
  // unused segment capacity stays zero, like the host planner's memset
  const int64_t cap = items + n;
  for (int64_t j = nseg + tid; j < cap; j += kPlanThreads) segs[j] = make_int4(0, 0, 0, 0);
  for (int64_t j = PH_WORDS + tid; j < off.cta_off; j += kPlanThreads) plan[j] = 0;
  for (int64_t j = off.cta_off + n + 1 + tid; j < off.segs; j += kPlanThreads) plan[j] = 0;
  if (tid == 0) {
    for (int j = 0; j < PH_WORDS; ++j) plan[j] = 0;
    plan[PH_MAGIC] = kPlanMagic;
    plan[PH_BATCH] = batch;
    plan[PH_NGRP] = ngrp;
    plan[PH_NCTAS] = n;
    plan[PH_GRANULE] = kGranule;
    plan[PH_NITEMS] = int(items);
    plan[PH_NSEGS] = nseg;
    plan[PH_NSLOTS] = nslots;
    plan[PH_TOTAL] = int(total);
    plan[PH_MODE] = SKD_PLAN_STREAMK;
    plan[PH_SEGCAP] = int(cap);
    plan[PH_ERR] = 0;
    plan[PH_SEGCOST] = seg_cost;
    plan[PH_ALIGN] = align;
  }
}

}  // namespace

int launch_plan_device(const int32_t *seqlens, int batch, int ngrp, int n, int seg_cost, int align, int32_t *plan,
                       cudaStream_t stream) {
  if (seg_cost < 0 || seg_cost > kMaxSegCost || align < 1 || align > kMaxAlign) return SKD_EINVAL;
  const size_t smem = size_t(batch + 1 + 2 * (n + 1)) * 4;
  if (smem > 200 * 1024) return SKD_EUNSUPPORTED;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(plan_device_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem)) != cudaSuccess)
    return SKD_ECUDA;
  plan_device_kernel<<<1, kPlanThreads, smem, stream>>>(seqlens, batch, ngrp, n, seg_cost, align, plan);
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace skd
