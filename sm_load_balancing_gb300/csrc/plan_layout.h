// Binary layout of a decode plan (int32 words). Shared by the host planner,
// the device planner and the kernels of this library only.
//
//   [0, 16)                  header (PH_*)
//   cta_seg_offset[n+1]      segments of CTA c are [off[c], off[c+1])
//   segs[cap][4]             {item, tok_begin, tok_end, slot}, 16-byte aligned;
//                            item = b*NGRP + g (g = kv-head group); slot = -1 when the segment is the
//                            whole item, else its workspace slot for partials
//   item_nsplit[num_items]   number of segments of each item
//   item_slot0[num_items]    slot of split 0 (splits use consecutive slots)
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define SKD_HD __host__ __device__
#else
#define SKD_HD
#endif

namespace skd {

// kv heads handled together by one CTA: the largest divisor of Hkv not above 8
SKD_HD inline int head_group(int hkv) {
  for (int g = hkv < 8 ? hkv : 8; g > 1; --g)
    if (hkv % g == 0) return g;
  return 1;
}

constexpr int32_t kPlanMagic = 0x534B4431;  // "SKD1"
constexpr int kGranule = 16;
constexpr int kMaxSegCost = 1 << 16;  // granules
constexpr int kMaxAlign = 64;         // granules per cut unit

enum PlanHeader : int {
  PH_MAGIC = 0,
  PH_BATCH = 1,
  PH_NGRP = 2,  // work items per request (kv-head groups)
  PH_NCTAS = 3,
  PH_GRANULE = 4,
  PH_NITEMS = 5,
  PH_NSEGS = 6,
  PH_NSLOTS = 7,
  PH_TOTAL = 8,  // total cut units (granules x PH_ALIGN)
  PH_MODE = 9,
  PH_SEGCAP = 10,
  PH_ERR = 11,  // device planner's error bits (SKD_DEVERR_*), 0 from the host planner
  PH_SEGCOST = 12,  // virtual granules charged per non-empty item (0: plain split)
  PH_ALIGN = 13,    // granules per cut unit: split points fall on multiples of kGranule * PH_ALIGN tokens
  PH_WORDS = 16
};

struct PlanOffsets {
  int64_t cta_off, segs, nsplit, slot0, words;
};

SKD_HD inline int64_t align4(int64_t x) { return (x + 3) & ~int64_t(3); }

SKD_HD inline PlanOffsets plan_offsets(int batch, int hkv, int n_ctas) {
  PlanOffsets o;
  int64_t items = int64_t(batch) * hkv;
  int64_t cap = items + n_ctas;
  o.cta_off = PH_WORDS;
  o.segs = o.cta_off + align4(int64_t(n_ctas) + 1);
  o.nsplit = o.segs + 4 * cap;
  o.slot0 = o.nsplit + items;
  o.words = o.slot0 + items;
  return o;
}

}  // namespace skd
