// Stream-K split-KV GQA decode attention for sm_103a.
//
// One persistent wave: CTA c walks the segment list the planner gave it (a
// near-equal share of the batch's KV tokens; triton.csdn.net Q&A on waves and
// FlashMLA's Stream-K, closing summary). Per segment (request b, kv head h,
// token range) the CTA streams paged K/V with TMA and keeps an online softmax
// ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 6.3 / Q8:
// QK^T -> mask -> softmax -> xV without writing scores to HBM). A segment that
// is only part of its (b, h) item writes its partial state (m, l, acc) to an
// L2-resident workspace slot and bumps the item's arrival counter; the split
// that arrives last merges all partials of the item right there
// ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", core method:
// just-in-time reduction, no separate reduction kernel and no wait for the
// slowest split). Nobody ever waits for another CTA, so the kernel is correct
// for any grid size and any scheduling order.
//
// CTA layout: warps 0..3 consume, warp 4 (one lane) produces.
//   stage  = 64 tokens of one kv head: K and V tiles, each D/64 sub-tiles of
//            [64 rows][128 B] with the 128-byte TMA swizzle;
//   warp w = the w-th 16-token granule of every stage; it keeps its own
//            (m, l, O) for the rows of the item and the four warps are merged
//            in shared memory at the end of the segment.
//   rows   = the G*T query rows sharing kv head h (padded to 16 for
//            mma.sync m16n8k16; row r is query token r / G, head h*G + r % G).
#include <math.h>

#include "kernels.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace skd {
namespace {

constexpr int kBlockN = 64;
constexpr int kCWarps = 4;
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kCThreads = kCWarps * 32;

template <int D>
struct Smem {
  static constexpr int kStages = 4;
  static constexpr int kSub = D / 64;
  static constexpr int kSubBytes = kBlockN * 128;
  static constexpr int kTileBytes = kSub * kSubBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
  static constexpr int kQBytes = 16 * D * 2;
  static constexpr int kOStride = D + 8;  // floats; padding keeps fragment stores conflict-free
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kOOff = kQOff + 2 * kQBytes;
  static constexpr int kMOff = kOOff + kCWarps * 16 * kOStride * 4;
  static constexpr int kLOff = kMOff + kCWarps * 16 * 4;   // sum of bf16-rounded p
  static constexpr int kLfOff = kLOff + kCWarps * 16 * 4;  // sum of fp32 p
  static constexpr int kBarOff = kLfOff + kCWarps * 16 * 4;
  static constexpr int kNumBars = 2 * kStages + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Params {
  const __nv_bfloat16 *q;
  const int32_t *page_table;
  const int32_t *seqlens;
  const int32_t *plan;
  int32_t *err;
  int32_t *counters;
  float *partials;
  __nv_bfloat16 *out;
  float *lse;
  int batch, T, Hq, Hkv, G, P, max_pages, num_pages, causal, rows, max_slots;
  float scale_log2;
  int64_t slot_floats;
};

__device__ __forceinline__ float fmax4(float a, float b, float c, float d) {
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const Params p) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t *plan = p.plan;

  // A plan built for another launch is rejected by every thread alike.
  if (plan[PH_MAGIC] != kPlanMagic || plan[PH_BATCH] != p.batch || plan[PH_HKV] != p.Hkv ||
      plan[PH_NCTAS] != int(gridDim.x) || plan[PH_GRANULE] != kGranule ||
      plan[PH_NSLOTS] > p.max_slots || plan[PH_ERR] != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, plan[PH_ERR] != 0 ? plan[PH_ERR] : SKD_DEVERR_PLAN);
    return;
  }
  const PlanOffsets off = plan_offsets(p.batch, p.Hkv, gridDim.x);
  const int seg_lo = plan[off.cta_off + blockIdx.x];
  const int seg_hi = plan[off.cta_off + blockIdx.x + 1];
  const int4 *segs = reinterpret_cast<const int4 *>(plan + off.segs);

  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + S::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S::kStages + s); };
  auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * S::kStages + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * S::kStages + 2 + s); };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kMiscOff);
  volatile int *last_flag = abort_flag + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), kCWarps);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(qfull_bar(s), 1);
      ptx::mbar_init(qempty_bar(s), kCWarps);
    }
    *abort_flag = 0;
    *last_flag = 0;
    ptx::fence_mbar_init();
  }
  // Q slots: rows beyond G*T stay zero for the whole kernel.
  {
    int4 *qz = reinterpret_cast<int4 *>(smem + S::kQOff);
    for (int i = threadIdx.x; i < 2 * S::kQBytes / 16; i += kThreads) qz[i] = make_int4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();

  const int Hkv = p.Hkv, G = p.G, T = p.T, rows = p.rows;

  // =========================== producer ====================================
  if (warp == kCWarps) {
    if (lane != 0) return;
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    const uint64_t pol = ptx::policy_evict_first();
    int stage = 0, qs = 0;
    uint32_t phase = 0, qph = 0;
    uint32_t last_parity_mask = 0, used_mask = 0;  // for the final drain
    bool ok = true;
    for (int si = seg_lo; si < seg_hi && ok; ++si) {
      const int4 sg = segs[si];
      const int item = sg.x, tb = sg.y, te = sg.z;
      if (te <= tb) continue;
      const int b = item / Hkv, h = item - b * Hkv;
      const int L = p.seqlens[b];
      if (te > L || L > p.max_pages * p.P || (p.causal && L < T)) atomicOr(p.err, SKD_DEVERR_SEQLEN);
      if (!ptx::mbar_wait(qempty_bar(qs), qph ^ 1u, abort_flag, kWaitCycles)) {
        ok = false;
        break;
      }
      ptx::mbar_arrive_expect_tx(qfull_bar(qs), uint32_t(rows * D * 2));
      for (int t = 0; t < T; ++t) {
        const __nv_bfloat16 *src = p.q + ((int64_t(b) * T + t) * p.Hq + int64_t(h) * G) * D;
        ptx::bulk_load(sbase + S::kQOff + qs * S::kQBytes + t * G * D * 2, src, uint32_t(G * D * 2),
                       qfull_bar(qs));
      }
      if (++qs == 2) {
        qs = 0;
        qph ^= 1u;
      }
      const int32_t *ptab = p.page_table + int64_t(b) * p.max_pages;
      for (int tok0 = tb; tok0 < te; tok0 += kBlockN) {
        if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
        const int ng = min(kBlockN / kGranule, (te - tok0 + kGranule - 1) / kGranule);
        ptx::mbar_arrive_expect_tx(full_bar(stage), uint32_t(ng * kGranule * 2 * D * 2));
        const uint32_t kdst = sbase + stage * S::kStageBytes;
        const uint32_t vdst = kdst + S::kTileBytes;
        for (int gi = 0; gi < ng; ++gi) {
          const int tok = tok0 + gi * kGranule;
          const int j = tok / p.P, slot = tok - j * p.P;
          int pg = j < p.max_pages ? ptab[j] : -1;
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.err, SKD_DEVERR_PAGE);
            pg = 0;
          }
#pragma unroll
          for (int sub = 0; sub < S::kSub; ++sub) {
            const uint32_t o = sub * S::kSubBytes + gi * kGranule * 128;
            ptx::tma_load_4d(kdst + o, &tmK, full_bar(stage), sub * 64, h, slot, pg, pol);
            ptx::tma_load_4d(vdst + o, &tmV, full_bar(stage), sub * 64, h, slot, pg, pol);
          }
        }
        used_mask |= 1u << stage;
        last_parity_mask = (last_parity_mask & ~(1u << stage)) | (phase << stage);
        if (++stage == S::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) *abort_flag = 1, atomicOr(p.err, SKD_DEVERR_TIMEOUT);
    // Drain: every fill this thread issued must have landed before the CTA
    // may exit (normally the consumers have already waited for all of them).
    for (int s = 0; s < S::kStages; ++s)
      if (used_mask & (1u << s))
        ptx::mbar_wait(full_bar(s), (last_parity_mask >> s) & 1u, nullptr, kWaitCycles);
    return;
  }

  // =========================== consumers ===================================
  const int w = warp;
  const int tid = threadIdx.x;  // 0..127
  const int fr = lane >> 2;     // fragment row (and row + 8)
  const int fc = lane & 3;      // fragment column pair
  float *sm_o = reinterpret_cast<float *>(smem + S::kOOff);
  float *sm_m = reinterpret_cast<float *>(smem + S::kMOff);
  float *sm_l = reinterpret_cast<float *>(smem + S::kLOff);
  float *sm_lf = reinterpret_cast<float *>(smem + S::kLfOff);
  const float NEG_INF = -INFINITY;
  int stage = 0, qs = 0;
  uint32_t phase = 0, qph = 0;

  for (int si = seg_lo; si < seg_hi; ++si) {
    const int4 sg = segs[si];
    const int item = sg.x, tb = sg.y, te = sg.z, wslot = sg.w;
    const int b = item / Hkv, h = item - b * Hkv;
    // combine-phase mapping: thread -> (row, 1/8 of the columns)
    const int cr = tid >> 3;
    const int cb = (tid & 7) * (D / 8);
    const int ct = cr < rows ? cr / G : 0;
    const int64_t orow = ((int64_t(b) * T + ct) * p.Hq + int64_t(h) * G + (cr - ct * G));

    if (te <= tb) {  // empty request: out = 0, lse = -inf
      if (cr < rows) {
        int4 *o4 = reinterpret_cast<int4 *>(p.out + orow * D + cb);
#pragma unroll
        for (int i = 0; i < D / 64; ++i) o4[i] = make_int4(0, 0, 0, 0);
        if ((tid & 7) == 0) p.lse[orow] = NEG_INF;
      }
      continue;
    }
    const int L = p.seqlens[b];

    // ---- Q fragments (A operand, rows x D) ----
    uint32_t qa[D / 16][4];
    bool alive = !*abort_flag;
    if (alive && !ptx::mbar_wait(qfull_bar(qs), qph, abort_flag, kWaitCycles)) {
      alive = false;
      *abort_flag = 1;
    }
    if (alive) {
      const uint32_t qb = sbase + S::kQOff + qs * S::kQBytes;
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ptx::ldsm_x4(qb + r * D * 2 + (2 * kk + (lane >> 4)) * 16, qa[kk][0], qa[kk][1], qa[kk][2],
                     qa[kk][3]);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(qempty_bar(qs));
    if (++qs == 2) {
      qs = 0;
      qph ^= 1u;
    }

    // last visible key of fragment rows fr and fr + 8 (causal: L - T + t)
    const int r0 = fr, r1 = fr + 8;
    const int lim0 = (p.causal && r0 < rows) ? L - T + r0 / G : INT_MAX;
    const int lim1 = (p.causal && r1 < rows) ? L - T + r1 / G : INT_MAX;

    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    // l: sum of the bf16-rounded p that enter P.V (normalises out, so out is an
    // exact convex combination of V rows); lf: sum of fp32 p (gives lse)
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f, lf0 = 0.f, lf1 = 0.f;

    for (int tok0 = tb; tok0 < te; tok0 += kBlockN) {
      if (alive && !ptx::mbar_wait(full_bar(stage), phase, abort_flag, kWaitCycles)) {
        alive = false;
        *abort_flag = 1;
      }
      const int mytok = tok0 + w * kGranule;
      if (alive && mytok < te) {
        const uint32_t kb = sbase + stage * S::kStageBytes;
        const uint32_t vb = kb + S::kTileBytes;
        if (mytok + kGranule > te) {
          // rows past the end of the request hold arbitrary bytes: zero their V
          const int r_lo = te - mytok;
          const int chunks = (kGranule - r_lo) * S::kSub * 8;
          for (int c = lane; c < chunks; c += 32) {
            const int rr = r_lo + c / (S::kSub * 8);
            const int rest = c % (S::kSub * 8);
            const int sub = rest >> 3, ch = rest & 7;
            int4 *dst = reinterpret_cast<int4 *>(smem + stage * S::kStageBytes + S::kTileBytes +
                                                 sub * S::kSubBytes + (w * kGranule + rr) * 128 +
                                                 ch * 16);
            *dst = make_int4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
        }
        // ---- S = Q K^T over this warp's 16 tokens ----
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int trow = w * kGranule + ((lane >> 4) << 3) + (lane & 7);
          const uint32_t rbase = kb + trow * 128;
          const int sw = trow & 7;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int ch = 2 * (kk & 3) + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4(rbase + (kk >> 2) * S::kSubBytes + ((ch ^ sw) << 4), b0, b1, b2, b3);
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
            const int tok = mytok + 8 * j + 2 * fc + e;
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
          const int trow = w * kGranule + (lane & 7) + (((lane >> 3) & 1) << 3);
          const uint32_t rbase = vb + trow * 128;
          const int sw = trow & 7;
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj) {
            const int chg = 2 * jj + (lane >> 4);  // 8-column chunk of V
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4_t(rbase + (chg >> 3) * S::kSubBytes + (((chg & 7) ^ sw) << 4), b0, b1, b2,
                           b3);
            ptx::mma_bf16_16816(o[2 * jj], pa, b0, b1);
            ptx::mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty_bar(stage));
      if (++stage == S::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- merge the four warps' states of this segment ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    lf0 += __shfl_xor_sync(0xffffffffu, lf0, 1);
    lf0 += __shfl_xor_sync(0xffffffffu, lf0, 2);
    lf1 += __shfl_xor_sync(0xffffffffu, lf1, 1);
    lf1 += __shfl_xor_sync(0xffffffffu, lf1, 2);
    if (fc == 0) {
      sm_m[w * 16 + r0] = m0;
      sm_m[w * 16 + r1] = m1;
      sm_l[w * 16 + r0] = l0;
      sm_l[w * 16 + r1] = l1;
      sm_lf[w * 16 + r0] = lf0;
      sm_lf[w * 16 + r1] = lf1;
    }
    {
      float *ow = sm_o + w * 16 * S::kOStride;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        *reinterpret_cast<float2 *>(ow + r0 * S::kOStride + 8 * j + 2 * fc) = make_float2(o[j][0], o[j][1]);
        *reinterpret_cast<float2 *>(ow + r1 * S::kOStride + 8 * j + 2 * fc) = make_float2(o[j][2], o[j][3]);
      }
    }
    ptx::named_bar(1, kCThreads);

    const bool split = wslot >= 0;
    const bool live = !*abort_flag;
    float acc[D / 8];
    float M = NEG_INF, Lt = 0.f, Lf = 0.f;
    if (cr < rows && live) {
#pragma unroll
      for (int ww = 0; ww < kCWarps; ++ww) M = fmaxf(M, sm_m[ww * 16 + cr]);
      const float Mu = M == NEG_INF ? 0.f : M;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) acc[c] = 0.f;
#pragma unroll
      for (int ww = 0; ww < kCWarps; ++ww) {
        const float f = exp2f(sm_m[ww * 16 + cr] - Mu);
        Lt += sm_l[ww * 16 + cr] * f;
        Lf += sm_lf[ww * 16 + cr] * f;
        const float *src = sm_o + (ww * 16 + cr) * S::kOStride + cb;
#pragma unroll
        for (int c = 0; c < D / 8; c += 4) {
          const float4 v = *reinterpret_cast<const float4 *>(src + c);
          acc[c] += v.x * f;
          acc[c + 1] += v.y * f;
          acc[c + 2] += v.z * f;
          acc[c + 3] += v.w * f;
        }
      }
      if (!split) {
        const float inv = 1.f / Lt;
        uint32_t pk[D / 16];
#pragma unroll
        for (int c = 0; c < D / 8; c += 2) pk[c / 2] = ptx::pack_bf16(acc[c] * inv, acc[c + 1] * inv);
        int4 *o4 = reinterpret_cast<int4 *>(p.out + orow * D + cb);
#pragma unroll
        for (int i = 0; i < D / 64; ++i) o4[i] = make_int4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        if ((tid & 7) == 0) p.lse[orow] = (M + log2f(Lf)) * 0.69314718055994531f;
      } else {
        float *ps = p.partials + int64_t(wslot) * p.slot_floats;
        float4 *d4 = reinterpret_cast<float4 *>(ps + cr * D + cb);
#pragma unroll
        for (int c = 0; c < D / 8; c += 4) d4[c / 4] = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        if ((tid & 7) == 0) {
          ps[rows * D + cr] = M;
          ps[rows * D + rows + cr] = Lt;
          ps[rows * D + 2 * rows + cr] = Lf;
        }
      }
    }
    if (split) {
      // publish the partial, count arrivals; the last split merges
      __threadfence();
      ptx::named_bar(1, kCThreads);
      if (tid == 0) {
        int last = 0;
        if (!*abort_flag) {
          const int nsp = plan[off.nsplit + item];
          const int old = atomicAdd(p.counters + item, 1);
          last = (old == nsp - 1) ? 1 : 0;
        }
        *last_flag = last;
      }
      ptx::named_bar(1, kCThreads);
      if (*last_flag) {
        __threadfence();
        const int nsp = plan[off.nsplit + item];
        const int s0 = plan[off.slot0 + item];
        if (cr < rows) {
          float Mx = NEG_INF;
          for (int s = 0; s < nsp; ++s)
            Mx = fmaxf(Mx, __ldcg(p.partials + int64_t(s0 + s) * p.slot_floats + rows * D + cr));
          const float Mu = Mx == NEG_INF ? 0.f : Mx;
          float lam = 0.f, lamf = 0.f;
#pragma unroll
          for (int c = 0; c < D / 8; ++c) acc[c] = 0.f;
          for (int s = 0; s < nsp; ++s) {
            const float *ps = p.partials + int64_t(s0 + s) * p.slot_floats;
            const float f = exp2f(__ldcg(ps + rows * D + cr) - Mu);
            lam += __ldcg(ps + rows * D + rows + cr) * f;
            lamf += __ldcg(ps + rows * D + 2 * rows + cr) * f;
            const float4 *src = reinterpret_cast<const float4 *>(ps + cr * D + cb);
#pragma unroll
            for (int c = 0; c < D / 8; c += 4) {
              const float4 v = __ldcg(src + c / 4);
              acc[c] += v.x * f;
              acc[c + 1] += v.y * f;
              acc[c + 2] += v.z * f;
              acc[c + 3] += v.w * f;
            }
          }
          const float inv = 1.f / lam;
          uint32_t pk[D / 16];
#pragma unroll
          for (int c = 0; c < D / 8; c += 2) pk[c / 2] = ptx::pack_bf16(acc[c] * inv, acc[c + 1] * inv);
          int4 *o4 = reinterpret_cast<int4 *>(p.out + orow * D + cb);
#pragma unroll
          for (int i = 0; i < D / 64; ++i)
            o4[i] = make_int4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          if ((tid & 7) == 0) p.lse[orow] = (Mx + log2f(lamf)) * 0.69314718055994531f;
        }
        if (tid == 0) p.counters[item] = 0;
      }
    }
    ptx::named_bar(1, kCThreads);  // shared scratch is reused by the next segment
  }
}

template <int D>
int launch_d(const DecodeArgs &a) {
  using S = Smem<D>;
  const skd_shape_t &s = a.shape;
  CUtensorMap tk, tv;
  const cuuint64_t gk[4] = {cuuint64_t(D), cuuint64_t(s.num_kv_heads), cuuint64_t(s.page_size),
                            cuuint64_t(s.num_pages)};
  const cuuint64_t sk[3] = {cuuint64_t(D) * 2, cuuint64_t(s.num_kv_heads) * D * 2,
                            cuuint64_t(s.page_size) * s.num_kv_heads * D * 2};
  const cuuint64_t sv[3] = {cuuint64_t(s.v_row_stride) * 2, cuuint64_t(s.num_kv_heads) * s.v_row_stride * 2,
                            cuuint64_t(s.page_size) * s.num_kv_heads * s.v_row_stride * 2};
  const cuuint32_t box[4] = {64, 1, cuuint32_t(kGranule), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.k), gk, sk, box, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return SKD_EINVAL;
  if (encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.v), gk, sv, box, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return SKD_EINVAL;

  Params p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.page_table = a.page_table;
  p.seqlens = a.seqlens;
  p.plan = a.plan;
  p.err = static_cast<int32_t *>(a.ws);
  p.counters = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(a.ws) + a.wl.counters);
  p.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(a.ws) + a.wl.partials);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.batch = s.batch;
  p.T = s.q_tokens;
  p.Hq = s.num_q_heads;
  p.Hkv = s.num_kv_heads;
  p.G = s.num_q_heads / s.num_kv_heads;
  p.P = s.page_size;
  p.max_pages = s.max_pages_per_req;
  p.num_pages = s.num_pages;
  p.causal = s.causal ? 1 : 0;
  p.rows = p.G * s.q_tokens;
  p.max_slots = int(a.wl.slots);
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.slot_floats = a.wl.slot_floats;

  static bool attr_set = false;  // per-process; the attribute is per function
  if (!attr_set) {
    if (cudaFuncSetAttribute(gqa_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kAlloc) != cudaSuccess)
      return SKD_ECUDA;
    attr_set = true;
  }
  gqa_decode_kernel<D><<<a.n_ctas, kThreads, S::kAlloc, a.stream>>>(tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace

int launch_gqa(const DecodeArgs &a) {
  const int D = a.shape.head_dim_qk;
  if (a.shape.head_dim_v != D) return SKD_EUNSUPPORTED;
  if ((a.shape.num_q_heads / a.shape.num_kv_heads) * a.shape.q_tokens > 16) return SKD_EUNSUPPORTED;
  if (D == 128) return launch_d<128>(a);
  if (D == 64) return launch_d<64>(a);
  return SKD_EUNSUPPORTED;
}

}  // namespace skd
