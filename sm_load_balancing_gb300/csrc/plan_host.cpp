// Host planner: the Stream-K one-wave split of a decode batch.
//
// "传统 GEMM 计算可能因任务大小不均产生多个调度波次（Waves）..." (triton.csdn.net Q&A
// on waves and FlashMLA's Stream-K), closing summary: cut the total work into
// exactly as many near-equal chunks as there are SMs and launch one wave, so no
// tail wave waits on a slow CTA. "MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）",
// core method: the mapping is decided at run time from the actual lengths.
//
// Work item i = b*NGRP + g (kv-head group g) carries ceil(L_b / 16) granules; CTA c receives the
// granule range [floor(c*G/n), floor((c+1)*G/n)) of the items laid end to end,
// cut at item boundaries. A single linear sweep, O(items + n).
//
// Optional segment cost (an extension beyond the pages): every non-empty item
// is preceded by `seg_cost` virtual granules that carry no tokens, standing for
// the fixed work a CTA spends per segment (loading the item's queries, writing
// its output or partial state). The equal split then runs over the virtual
// total, so a CTA that crosses many item boundaries receives fewer tokens.
// seg_cost = 0 is the plain split.
//
// Optional alignment (also an extension): with align > 1 the split runs over
// cut units of align granules, so split points fall on multiples of
// kGranule * align tokens of an item (a kernel that reads whole blocks of that
// many tokens then never reads a block twice), and the segment cost is
// ceil(seg_cost / align) units. align = 1 is the plan above.
#include <string.h>

#include <vector>

#include "plan_layout.h"
#include "skdecode.h"

namespace skd {

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int build_plan_host(const int32_t *seqlens, int batch, int ngrp, int page_size, int n, int mode,
                    int seg_cost, int align, void *plan_out, size_t plan_bytes) {
  if (!seqlens && batch > 0) return SKD_EINVAL;
  if (!plan_out || batch < 0 || ngrp <= 0 || n <= 0) return SKD_EINVAL;
  if (page_size <= 0 || page_size % kGranule != 0) return SKD_EINVAL;
  if (mode != SKD_PLAN_STREAMK && mode != SKD_PLAN_ROUND_ROBIN && mode != SKD_PLAN_FIXED_SPLIT) return SKD_EINVAL;
  if (seg_cost < 0 || seg_cost > kMaxSegCost || (seg_cost > 0 && mode != SKD_PLAN_STREAMK)) return SKD_EINVAL;
  if (align < 1 || align > kMaxAlign || (align > 1 && mode != SKD_PLAN_STREAMK)) return SKD_EINVAL;
  const int64_t unit = int64_t(kGranule) * align;                // tokens per cut unit
  const int64_t vcost = ceil_div(seg_cost, align);               // virtual units per item
  const PlanOffsets off = plan_offsets(batch, ngrp, n);
  if (plan_bytes < size_t(off.words) * 4) return SKD_EPLAN;
  for (int b = 0; b < batch; ++b)
    if (seqlens[b] < 0) return SKD_EINVAL;

  const int64_t items = int64_t(batch) * ngrp;
  const int64_t cap = items + n;
  int32_t *w = static_cast<int32_t *>(plan_out);
  memset(w, 0, size_t(off.words) * 4);
  int32_t *cta_off = w + off.cta_off;
  int32_t *segs = w + off.segs;
  int32_t *nsplit = w + off.nsplit;
  int32_t *slot0 = w + off.slot0;

  int64_t total = 0;  // virtual cut units (granules when align = 1)
  for (int b = 0; b < batch; ++b) {
    const int64_t g = ceil_div(seqlens[b], unit);
    total += int64_t(ngrp) * (g + (g > 0 ? vcost : 0));
  }
  if (total > INT32_MAX) return SKD_EPLAN;

  int64_t nseg = 0;
  auto push = [&](int64_t item, int64_t tb, int64_t te) {
    int32_t *s = segs + 4 * nseg;
    s[0] = int32_t(item);
    s[1] = int32_t(tb);
    s[2] = int32_t(te);
    s[3] = -1;
    ++nseg;
  };

  if (mode == SKD_PLAN_STREAMK) {
    auto bound = [&](int64_t c) { return (c * total) / n; };
    int64_t c = 0, pos = 0;
    cta_off[0] = 0;
    auto close_ctas_up_to = [&](int64_t cnew) {
      // CTAs c .. cnew-1 are complete: record where CTA c+1.. begins
      while (c < cnew) {
        ++c;
        cta_off[c] = int32_t(nseg);
      }
    };
    for (int64_t i = 0; i < items; ++i) {
      const int64_t L = seqlens[i / ngrp];
      const int64_t g = ceil_div(L, unit);
      // token units of the item occupy [s, e) after its virtual segment cost
      const int64_t s = pos + (g > 0 ? vcost : 0), e = s + g;
      pos = e;
      // first CTA whose chunk ends after s (the last CTA if none)
      int64_t cs = c;
      while (cs < n - 1 && bound(cs + 1) <= s) ++cs;
      close_ctas_up_to(cs);
      if (g == 0) {
        push(i, 0, 0);
        continue;
      }
      for (int64_t cc = cs; cc < n; ++cc) {
        const int64_t lo = s > bound(cc) ? s : bound(cc);
        const int64_t hi = e < bound(cc + 1) ? e : bound(cc + 1);
        if (lo >= hi) {
          if (bound(cc) >= e) break;
          continue;
        }
        close_ctas_up_to(cc);
        const int64_t tb = (lo - s) * unit;
        const int64_t te = (hi - s) * unit < L ? (hi - s) * unit : L;
        push(i, tb, te);
      }
    }
    close_ctas_up_to(n);
    cta_off[n] = int32_t(nseg);
  } else if (mode == SKD_PLAN_FIXED_SPLIT) {
    // the two-kernel comparator: every item cut into S = max(1, floor(n /
    // items)) near-equal granule ranges (fewer if it has fewer granules), so
    // that all splits fill about one wave; split j of the whole list goes to
    // CTA j mod n, like a grid of (item, split) blocks
    const int64_t S = items > 0 ? (n / items > 1 ? n / items : 1) : 1;
    std::vector<int32_t> all;  // (item, tb, te, slot) in item / split order
    int64_t slots = 0;
    for (int64_t i = 0; i < items; ++i) {
      const int64_t L = seqlens[i / ngrp];
      const int64_t g = ceil_div(L, kGranule);
      const int64_t s = g < S ? (g > 0 ? g : 1) : S;
      nsplit[i] = int32_t(s);
      slot0[i] = s > 1 ? int32_t(slots) : -1;
      for (int64_t k = 0; k < s; ++k) {
        const int64_t lo = (k * g) / s, hi = ((k + 1) * g) / s;
        all.push_back(int32_t(i));
        all.push_back(int32_t(lo * kGranule));
        all.push_back(int32_t(hi * kGranule < L ? hi * kGranule : L));
        all.push_back(s > 1 ? int32_t(slots + k) : -1);
      }
      if (s > 1) slots += s;
    }
    const int64_t total_segs = int64_t(all.size()) / 4;
    if (total_segs > cap) return SKD_EPLAN;
    for (int64_t c = 0; c < n; ++c) {
      cta_off[c] = int32_t(nseg);
      for (int64_t j = c; j < total_segs; j += n) {
        push(all[4 * j], all[4 * j + 1], all[4 * j + 2]);
        segs[4 * (nseg - 1) + 3] = all[4 * j + 3];
      }
    }
    cta_off[n] = int32_t(nseg);
  } else {
    // round robin: item i -> CTA i mod n, no splits
    for (int64_t c = 0; c < n; ++c) {
      cta_off[c] = int32_t(nseg);
      for (int64_t i = c; i < items; i += n) push(i, 0, seqlens[i / ngrp]);
    }
    cta_off[n] = int32_t(nseg);
  }
  if (nseg > cap) return SKD_EPLAN;  // cannot happen by construction

  // splits per item (segments of an item are consecutive in the list; the
  // fixed-split mode numbered its slots above)
  int64_t nslots = 0;
  if (mode == SKD_PLAN_FIXED_SPLIT)
    for (int64_t i = 0; i < items; ++i) nslots += nsplit[i] > 1 ? nsplit[i] : 0;
  for (int64_t k = 0; k < nseg && mode != SKD_PLAN_FIXED_SPLIT;) {
    const int32_t item = segs[4 * k];
    int64_t e = k;
    while (e < nseg && segs[4 * e] == item) ++e;
    const int64_t ns = e - k;
    nsplit[item] = int32_t(ns);
    slot0[item] = ns > 1 ? int32_t(nslots) : -1;
    if (ns > 1)
      for (int64_t j = k; j < e; ++j) segs[4 * j + 3] = int32_t(nslots++);
    k = e;
  }

  w[PH_MAGIC] = kPlanMagic;
  w[PH_BATCH] = batch;
  w[PH_NGRP] = ngrp;
  w[PH_NCTAS] = n;
  w[PH_GRANULE] = kGranule;
  w[PH_NITEMS] = int32_t(items);
  w[PH_NSEGS] = int32_t(nseg);
  w[PH_NSLOTS] = int32_t(nslots);
  w[PH_TOTAL] = int32_t(total);
  w[PH_MODE] = mode;
  w[PH_SEGCAP] = int32_t(cap);
  w[PH_ERR] = 0;
  w[PH_SEGCOST] = seg_cost;
  w[PH_ALIGN] = align;
  return SKD_OK;
}

}  // namespace skd
