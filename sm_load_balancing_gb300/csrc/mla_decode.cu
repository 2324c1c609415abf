// Absorbed-MLA decode attention on tcgen05 tensor cores (sm_103a).
//
// Shapes: 128 query heads share one latent KV row of 576 values per token;
// scores use all 576 columns, values are the first 512 ("GPU Kernel、异步
// Launch、Stream 与融合 Kernel 全解", section 6.3 / Q8: QK^T -> softmax -> xV
// fused on chip). Work is split Stream-K style across persistent workers
// (triton.csdn.net Q&A on waves and FlashMLA's Stream-K, closing summary) and
// partial states are merged just in time by the last split of each request
// ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", core method; its key
// observation that a cluster of SMs can cooperate through TMA/mbarrier is what
// the pair below uses).
//
// One worker = a 2-CTA cluster. TMEM holds 128 lanes x 512 fp32 columns: one
// 128x512 output accumulator, with no room for scores, and Q alone is 147 KB of
// shared memory, so the contraction is split over the pair:
//   rank 0 streams latent columns [0, 256), rank 1 columns [256, 576), one TMA
//   box per 64-token block each (no byte is read twice);
//   S = Q K^T: each rank computes the partial sum over its own columns
//   (M=128 heads, N=64 tokens) into TMEM and sends it to the partner over
//   DSMEM; both ranks add the two partials (same bits: addition commutes) and
//   run the same online softmax, one thread per head row;
//   O = P V: each rank accumulates its 256 value columns for all 128 heads in
//   TMEM (M=128, N=256, K=64 tokens) from its own copy of P.
// The running maximum is kept per row and only moved (with an O rescale) when
// a block's maximum exceeds it by more than 2^8, so p <= 256 and rescales are
// rare; l and O stay consistent with the same reference maximum.
// Every wait is bounded; a timeout sets the error word and an abort flag in
// both ranks so that the pair drains quickly.
#include <math.h>

#include <algorithm>

#include "kernels.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace skd {
namespace {

constexpr int kHeads = 128, kDk = 576, kDv = 512, kBlk = 64;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMaxSt = 4;
constexpr float kTau = 8.f;  // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kTraceWords = SKD_TRACE_RECORD_BYTES / 8;

// fixed shared-memory region (same offsets in both ranks, for DSMEM)
constexpr int kOffP = 0;                     // P [2 buffers][128 rows][64 tok] bf16, SW128: 32 KB
constexpr int kOffSx = 32768;                // partner's partial scores [128][64] fp32: 32 KB
constexpr int kOffBar = 65536;               // mbarriers
constexpr int kNumBar = 2 * kMaxSt + 20;
constexpr int kOffMisc = kOffBar + kNumBar * 8;  // tmem base, flags
constexpr int kOffQ = 65 * 1024;             // Q [nch][128][128 B], then KV stages

// barrier indices
// (P buffers alternate per block; B_PF*, B_PVD* and B_OR* come in pairs, one per
// buffer, so that no barrier can run two phases ahead of a waiter)
enum {
  B_KVF = 0, B_KVE = kMaxSt, B_QF = 2 * kMaxSt, B_QE, B_SF0, B_SF1, B_SE0, B_SE1, B_SXF, B_SXFREE,
  B_PF0, B_PF1, B_PVD0, B_PVD1, B_OR0, B_OR1, B_STF, B_PAIR, B_GO, B_FIN
};

struct Params {
  const int32_t *page_table;
  const int32_t *seqlens;
  const int32_t *plan;
  int32_t *err;
  int32_t *item_cnt;
  float *partials;
  __nv_bfloat16 *out;
  float *lse;
  int batch, P, max_pages, num_pages, max_slots, nst0, nst1;
  float scale_log2;
  int64_t slot_floats;
  long long *trace;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// UMMA shared-memory descriptor (128-byte swizzle): start, leading / stride byte offsets
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor, kind::f16: bf16 A/B, fp32 D, A K-major, B K- or MN-major
__host__ __device__ constexpr uint32_t idesc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void umma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// 32 lanes x 32 consecutive fp32 columns per warp (lane = TMEM lane of the warp's quarter)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1, int c2,
                                     uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}

struct Ctx {
  uint8_t *smem;
  uint32_t sbase, peer;  // own shared base; peer rank
  volatile int *abort;
  int32_t *err;
  __device__ uint32_t bar(int i) const { return sbase + kOffBar + 8u * i; }
  __device__ uint32_t peer_addr(uint32_t local) const { return mapa(local, peer); }
  // bounded wait with cluster-scope acquire; on timeout flag both ranks
  __device__ bool wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    if (try_wait_cluster(b, parity)) return true;
    const long long t0 = clock64();
    uint32_t n = 0;
    while (!try_wait_cluster(b, parity)) {
      if ((++n & 255u) == 0) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitCycles) {
          *abort = 1;
          st_cluster_u32(peer_addr(sbase + kOffMisc + 4), 1u);
          atomicOr(err, SKD_DEVERR_TIMEOUT);
          return false;
        }
      }
    }
    return true;
  }
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tq0, const __grid_constant__ CUtensorMap tq1,
                      const __grid_constant__ CUtensorMap tkv0, const __grid_constant__ CUtensorMap tkv1,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int worker = blockIdx.x >> 1;
  const int nworkers = gridDim.x >> 1;
  const int32_t *plan = p.plan;
  if (plan[PH_MAGIC] != kPlanMagic || plan[PH_BATCH] != p.batch || plan[PH_NGRP] != 1 ||
      plan[PH_NCTAS] != nworkers || plan[PH_GRANULE] != kGranule || plan[PH_NSLOTS] > p.max_slots ||
      plan[PH_ERR] != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, plan[PH_ERR] != 0 ? plan[PH_ERR] : SKD_DEVERR_PLAN);
    return;  // both ranks take this path alike
  }
  const PlanOffsets off = plan_offsets(p.batch, 1, nworkers);
  const int seg_lo = plan[off.cta_off + worker], seg_hi = plan[off.cta_off + worker + 1];
  const int4 *segs = reinterpret_cast<const int4 *>(plan + off.segs);

  const int nch = rank == 0 ? 4 : 5;              // 64-column chunks this rank streams
  const int chunk0 = rank == 0 ? 0 : 4;
  const int nst = rank == 0 ? p.nst0 : p.nst1;
  const uint32_t stage_bytes = uint32_t(nch) * kBlk * 128;
  const uint32_t q_bytes = uint32_t(nch) * kHeads * 128;
  const CUtensorMap *tq = rank == 0 ? &tq0 : &tq1;
  const CUtensorMap *tkv = rank == 0 ? &tkv0 : &tkv1;

  Ctx cx;
  cx.smem = smem;
  cx.sbase = ptx::smem_u32(smem);
  cx.peer = rank ^ 1u;
  cx.abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  cx.err = p.err;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  const uint32_t sQ = cx.sbase + kOffQ;
  const uint32_t sKV = sQ + q_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      ptx::mbar_init(cx.bar(B_KVF + s), 1);
      ptx::mbar_init(cx.bar(B_KVE + s), 1);
    }
    ptx::mbar_init(cx.bar(B_QF), 1);
    ptx::mbar_init(cx.bar(B_QE), 1);
    ptx::mbar_init(cx.bar(B_SF0), 1);
    ptx::mbar_init(cx.bar(B_SF1), 1);
    ptx::mbar_init(cx.bar(B_SE0), 4);
    ptx::mbar_init(cx.bar(B_SE1), 4);
    ptx::mbar_init(cx.bar(B_SXF), 4);
    ptx::mbar_init(cx.bar(B_SXFREE), 4);
    ptx::mbar_init(cx.bar(B_PF0), 4);
    ptx::mbar_init(cx.bar(B_PF1), 4);
    ptx::mbar_init(cx.bar(B_PVD0), 1);
    ptx::mbar_init(cx.bar(B_PVD1), 1);
    ptx::mbar_init(cx.bar(B_OR0), 4);
    ptx::mbar_init(cx.bar(B_OR1), 4);
    ptx::mbar_init(cx.bar(B_PAIR), 1);
    ptx::mbar_init(cx.bar(B_GO), 1);
    ptx::mbar_init(cx.bar(B_FIN), 1);
    *cx.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     cx.sbase + kOffMisc),
                 "r"(512u));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();  // barriers of both ranks initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS[2] = {tmem + 0, tmem + 64};  // partial / full scores, double buffered
  const uint32_t tO = tmem + 128;                 // this rank's 256 value columns

  // trace (when enabled): one record per CTA; words 2.. accumulate wait cycles
  long long *const tr = p.trace ? p.trace + int64_t(blockIdx.x) * kTraceWords : nullptr;
  if (tr && threadIdx.x == 0) tr[0] = (long long)ptx::globaltimer_ns();
  auto tw = [&](int idx, long long t0) {
    if (tr && lane == 0) atomicAdd(reinterpret_cast<unsigned long long *>(tr + idx), (unsigned long long)(clock64() - t0));
  };
  const long long tk0 = clock64();

  if (warp == 0) {
    // ============================ TMA producer ===============================
    const uint64_t pol = ptx::policy_evict_first();
    int st = 0, qn = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int si = seg_lo; si < seg_hi && ok; ++si) {
      const int4 sg = segs[si];
      const int b = sg.x, tb = sg.y, te = sg.z;
      if (te <= tb) continue;
      const int32_t *ptab = p.page_table + int64_t(b) * p.max_pages;
      if (lane == 0) {
        const int L = p.seqlens[b];
        if (te > L || L > p.max_pages * p.P) atomicOr(p.err, SKD_DEVERR_SEQLEN);
        ok = cx.wait(B_QE, (qn & 1) ^ 1u);
        if (ok) {
          ptx::mbar_arrive_expect_tx(cx.bar(B_QF), q_bytes);
          tma3(sQ, tq, cx.bar(B_QF), 0, b * kHeads, chunk0, pol);
        }
      }
      ++qn;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const int w_lo = (tb / kBlk) * kBlk;
      for (int w0 = w_lo; w0 < te && ok; w0 += kBlk) {
        if (lane == 0) {
          const int j = w0 / p.P;
          int pg = j < p.max_pages ? __ldg(ptab + j) : -1;
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.err, SKD_DEVERR_PAGE);
            pg = 0;
          }
          const long long t0 = clock64();
          ok = cx.wait(B_KVE + st, ph ^ 1u);
          tw(9, t0);
          if (ok) {
            ptx::mbar_arrive_expect_tx(cx.bar(B_KVF + st), stage_bytes);
            tma3(sKV + st * stage_bytes, tkv, cx.bar(B_KVF + st), 0, pg * p.P + (w0 % p.P), chunk0, pol);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (++st == nst) {
          st = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer =================================
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(kHeads, kBlk, 0);
      constexpr uint32_t id_pv = idesc(kHeads, 256, 1);
      int st = 0, qn = 0;
      uint32_t ph = 0;
      long long g = 0;  // global block counter (S buffers and per-block barriers)
      bool ok = true;
      for (int si = seg_lo; si < seg_hi && ok; ++si) {
        const int4 sg = segs[si];
        const int tb = sg.y, te = sg.z;
        if (te <= tb) continue;
        const int nb = (te + kBlk - 1) / kBlk - tb / kBlk;
        ok = cx.wait(B_QF, qn & 1);
        ++qn;
        tc_fence_after();
        auto issue_qk = [&](long long gg, int stage) {
          const int sb = int(gg & 1);
          const long long t0 = clock64();
          if (!cx.wait(sb ? B_SE1 : B_SE0, uint32_t(((gg >> 1) & 1) ^ 1))) return false;
          tw(8, t0);
          tc_fence_after();
          for (int c = 0; c < nch; ++c)
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc(sQ + c * (kHeads * 128) + kk * 32, 16, 1024);
              const uint64_t bd = sdesc(sKV + stage * stage_bytes + c * (kBlk * 128) + kk * 32, 16, 1024);
              umma(tS[sb], a, bd, id_qk, (c | kk) != 0);
            }
          umma_commit(cx.bar(sb ? B_SF1 : B_SF0));
          return true;
        };
        // block 0 of the segment
        int st_j = st;
        uint32_t ph_j = ph;
        ok = ok && cx.wait(B_KVF + st_j, ph_j);
        ok = ok && issue_qk(g, st_j);
        for (int j = 0; j < nb && ok; ++j) {
          // issue QK of block j+1 before waiting for the softmax of block j
          int st_n = st_j + 1;
          uint32_t ph_n = ph_j;
          if (st_n == nst) {
            st_n = 0;
            ph_n ^= 1u;
          }
          if (j + 1 < nb) {
            const long long t0 = clock64();
            ok = cx.wait(B_KVF + st_n, ph_n);
            tw(6, t0);
            ok = ok && issue_qk(g + 1, st_n);
            if (!ok) break;
          } else {
            umma_commit(cx.bar(B_QE));  // Q is free once this segment's last QK completes
          }
          // PV of block j (P buffer g & 1)
          const int pb = int(g & 1);
          const long long t0 = clock64();
          if (!cx.wait(B_PF0 + pb, uint32_t((g >> 1) & 1)) || !cx.wait(B_OR0 + pb, uint32_t((g >> 1) & 1))) {
            ok = false;
            break;
          }
          tw(7, t0);
          tc_fence_after();
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sdesc(cx.sbase + kOffP + pb * 16384 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(sKV + st_j * stage_bytes + kk * (16 * 128), kBlk * 128, 1024);
            umma(tO, a, bd, id_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(cx.bar(B_KVE + st_j));
          umma_commit(cx.bar(B_PVD0 + pb));
          st_j = st_n;
          ph_j = ph_n;
          ++g;
        }
        st = st_j;
        ph = ph_j;
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(cx.bar(B_FIN));
      cx.wait(B_FIN, 0);
    }
  } else {
    // ============================ epilogue warps =============================
    // Each rank computes the softmax of all 128 rows: it sends its partial
    // scores to the partner and adds the partner's, so both ranks hold the same
    // full scores (fp32 addition commutes) and derive the same P, rescale
    // factors and row statistics locally -- one exchange per block.
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;   // query head
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const float *sx = reinterpret_cast<const float *>(smem + kOffSx);
    long long g = 0;
    int pairn = 0;
    bool ok = true;
    for (int si = seg_lo; si < seg_hi; ++si) {
      const int4 sg = segs[si];
      const int b = sg.x, tb = sg.y, te = sg.z, wslot = sg.w;
      const int64_t orow = int64_t(b) * kHeads + row;
      if (te <= tb) {  // empty request
        uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + rank * 256);
        for (int c = 0; c < 32; ++c) o4[c] = make_uint4(0, 0, 0, 0);
        if (rank == 0) p.lse[orow] = -INFINITY;
        continue;
      }
      const int L = p.seqlens[b];
      const int nb = (te + kBlk - 1) / kBlk - tb / kBlk;
      float mref = -INFINITY, l = 0.f, lf = 0.f;
      for (int j = 0; j < nb; ++j, ++g) {
        const int w0 = (tb / kBlk) * kBlk + j * kBlk;
        const int sb = int(g & 1), pb = int(g & 1);
        float s[64];
        long long t0 = clock64();
        ok = ok && cx.wait(sb ? B_SF1 : B_SF0, uint32_t((g >> 1) & 1));
        tw(2, t0);
        if (tr && threadIdx.x == 64) atomicAdd(reinterpret_cast<unsigned long long *>(tr + 13), 1ull);
        tc_fence_after();
        tmem_ld32(tS[sb] + lane_off, s);
        tmem_ld32(tS[sb] + lane_off + 32, s + 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cx.bar(sb ? B_SE1 : B_SE0));
        // ---- exchange partial scores with the partner ----
        t0 = clock64();
        ok = ok && cx.wait(B_SXFREE, uint32_t((g & 1) ^ 1));
        const uint32_t dst = cx.peer_addr(cx.sbase + kOffSx + uint32_t(row) * 256);
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          st_cluster_v4(dst + c * 4, __float_as_uint(s[c]), __float_as_uint(s[c + 1]), __float_as_uint(s[c + 2]),
                        __float_as_uint(s[c + 3]));
        __syncwarp();
        if (lane == 0) arrive_remote(cx.peer_addr(cx.bar(B_SXF)));
        ok = ok && cx.wait(B_SXF, uint32_t(g & 1));
        tw(3, t0);
        {
          const float *mine = sx + row * 64;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(mine + c);
            s[c] += v.x;
            s[c + 1] += v.y;
            s[c + 2] += v.z;
            s[c + 3] += v.w;
          }
        }
        __syncwarp();
        if (lane == 0) arrive_remote(cx.peer_addr(cx.bar(B_SXFREE)));
        // ---- online softmax of this row (thread-local) ----
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int tok = w0 + c;
          s[c] = (tok >= tb && tok < te) ? s[c] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        float a = 1.f;
        if (j == 0) {
          mref = mx;
        } else if (mx > mref + kTau) {
          a = exp2f(mref - mx);
          mref = mx;
          l *= a;
          lf *= a;
        }
        uint32_t pk[32];
        float ps = 0.f, pf = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float e0 = exp2f(s[c] - mref), e1 = exp2f(s[c + 1] - mref);
          pf += e0 + e1;
          pk[c / 2] = ptx::pack_bf16(e0, e1);
          const float2 f = ptx::unpack_bf16(pk[c / 2]);
          ps += f.x + f.y;
        }
        l += ps;
        lf += pf;
        // P row into P buffer pb once PV(g-2), its previous reader, is done
        t0 = clock64();
        ok = ok && cx.wait(B_PVD0 + pb, uint32_t(((g >> 1) & 1) ^ 1));
        tw(4, t0);
        {
          const uint32_t prow = cx.sbase + kOffP + uint32_t(pb) * 16384 + uint32_t(row) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + uint32_t((c ^ (row & 7)) << 4)),
                         "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                         : "memory");
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cx.bar(B_PF0 + pb));
        // ---- rescale this rank's O columns if the max moved (rare) ----
        // (MMAs from one thread run in order, so without a rescale PV(g) may
        // follow PV(g-1) at once; a rescale first waits for PV(g-1) to finish)
        if (j > 0 && __any_sync(0xffffffffu, a != 1.f)) {
          t0 = clock64();
          ok = ok && cx.wait(B_PVD0 + int((g - 1) & 1), uint32_t(((g - 1) >> 1) & 1));
          tw(5, t0);
          tc_fence_after();
          float v[32];
          for (int c = 0; c < 256; c += 32) {
            tmem_ld32(tO + lane_off + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= a;
            tmem_st32(tO + lane_off + c, v);
          }
        }
        // rows of the block past the end of the request hold arbitrary bytes:
        // zero them in this rank's value chunks (the QK of this block is done)
        if (w0 + kBlk > L) {
          const int t_lo = L - w0;  // >= 1 because w0 < te <= L
          uint8_t *stage = smem + (sKV - cx.sbase) + uint32_t(g % nst) * stage_bytes;
          const int pieces = 4 * (kBlk - t_lo) * 8;
          for (int i = threadIdx.x - 64; i < pieces; i += 128) {
            const int c = i / ((kBlk - t_lo) * 8), rest = i - c * ((kBlk - t_lo) * 8);
            *reinterpret_cast<int4 *>(stage + c * (kBlk * 128) + (t_lo + (rest >> 3)) * 128 + (rest & 7) * 16) =
                make_int4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cx.bar(B_OR0 + pb));
      }
      // ---- segment end: wait for the last PV; this thread holds its row's stats ----
      ok = ok && cx.wait(B_PVD0 + int((g - 1) & 1), uint32_t(((g - 1) >> 1) & 1));
      tc_fence_after();
      if (wslot < 0) {
        const float inv = 1.f / l;
        float v[32];
        for (int c = 0; c < 256; c += 32) {
          tmem_ld32(tO + lane_off + c, v);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) pk[i / 2] = ptx::pack_bf16(v[i] * inv, v[i + 1] * inv);
          uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + rank * 256 + c);
#pragma unroll
          for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        if (rank == 0) p.lse[orow] = (mref + log2f(lf)) * kLn2;
      } else {
        float *ps = p.partials + int64_t(wslot) * p.slot_floats;
        float v[32];
        for (int c = 0; c < 256; c += 32) {
          tmem_ld32(tO + lane_off + c, v);
          float4 *d4 = reinterpret_cast<float4 *>(ps + row * kDv + rank * 256 + c);
#pragma unroll
          for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        if (rank == 0) {
          ps[kHeads * kDv + row] = mref;
          ps[kHeads * kDv + kHeads + row] = l;
          ps[kHeads * kDv + 2 * kHeads + row] = lf;
        }
      }
      tc_fence_before();
      // the O accumulator may be overwritten by the next segment's first PV
      __syncwarp();
      if (wslot >= 0) {
        // both ranks' partial writes, then one release-acquire arrival per pair
        const int nsp = plan[off.nsplit + b], s0 = plan[off.slot0 + b];
        ptx::named_bar(1, 128);
        int last = 0;
        if (rank == 1) {
          if (threadIdx.x == 64) {
            __threadfence();
            arrive_remote(cx.peer_addr(cx.bar(B_PAIR)));
          }
          ok = ok && cx.wait(B_GO, uint32_t(pairn & 1));
          last = *reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
        } else {
          if (threadIdx.x == 64) {
            int lst = 0;
            if (cx.wait(B_PAIR, uint32_t(pairn & 1)) && !*cx.abort)
              lst = ptx::atom_add_acq_rel_gpu(p.item_cnt + b, 1) == nsp - 1 ? 1 : 0;
            *reinterpret_cast<volatile int *>(smem + kOffMisc + 8) = lst;
            st_cluster_u32(cx.peer_addr(cx.sbase + kOffMisc + 8), uint32_t(lst));
            arrive_remote(cx.peer_addr(cx.bar(B_GO)));
            if (lst) p.item_cnt[b] = 0;
          }
          ptx::named_bar(1, 128);
          last = *reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
        }
        ++pairn;
        if (last) {
          // merge this rank's 256 columns of every split, in split order
          __threadfence();
          float Mx = -INFINITY;
          for (int s = 0; s < nsp; ++s)
            Mx = fmaxf(Mx, __ldcg(p.partials + int64_t(s0 + s) * p.slot_floats + kHeads * kDv + row));
          const float Mu = Mx == -INFINITY ? 0.f : Mx;
          float lam = 0.f, lamf = 0.f;
          for (int s = 0; s < nsp; ++s) {
            const float *ps = p.partials + int64_t(s0 + s) * p.slot_floats;
            const float f = exp2f(__ldcg(ps + kHeads * kDv + row) - Mu);
            lam += __ldcg(ps + kHeads * kDv + kHeads + row) * f;
            lamf += __ldcg(ps + kHeads * kDv + 2 * kHeads + row) * f;
          }
          const float inv = 1.f / lam;
          for (int c = 0; c < 256; c += 8) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int s = 0; s < nsp; ++s) {
              const float *ps = p.partials + int64_t(s0 + s) * p.slot_floats;
              const float f = exp2f(__ldcg(ps + kHeads * kDv + row) - Mu);
              const float4 *src = reinterpret_cast<const float4 *>(ps + row * kDv + rank * 256 + c);
              const float4 x = __ldcg(src), y = __ldcg(src + 1);
              acc[0] += x.x * f;
              acc[1] += x.y * f;
              acc[2] += x.z * f;
              acc[3] += x.w * f;
              acc[4] += y.x * f;
              acc[5] += y.y * f;
              acc[6] += y.z * f;
              acc[7] += y.w * f;
            }
            *reinterpret_cast<uint4 *>(p.out + orow * kDv + rank * 256 + c) =
                make_uint4(ptx::pack_bf16(acc[0] * inv, acc[1] * inv), ptx::pack_bf16(acc[2] * inv, acc[3] * inv),
                           ptx::pack_bf16(acc[4] * inv, acc[5] * inv), ptx::pack_bf16(acc[6] * inv, acc[7] * inv));
          }
          if (rank == 0) p.lse[orow] = (Mx + log2f(lamf)) * kLn2;
        }
      }
    }
    (void)ok;
  }
  // ---- teardown: both ranks leave together (the partner may still write here) ----
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u));
  }
  if (tr && lane == 0) {
    const int slot = warp == 0 ? 12 : (warp == 1 ? 11 : 10);
    atomicAdd(reinterpret_cast<unsigned long long *>(tr + slot), (unsigned long long)(clock64() - tk0));
  }
  if (tr && threadIdx.x == 0) {
    tr[14] = seg_hi - seg_lo;
    tr[15] = ptx::smid();
    tr[1] = (long long)ptx::globaltimer_ns();
  }
}

}  // namespace

int launch_mla(const DecodeArgs &a) {
  const skd_shape_t &s = a.shape;
  if (s.page_size % kBlk != 0) return SKD_EUNSUPPORTED;  // 64-token blocks must not straddle pages
  CUtensorMap tq[2], tkv[2];
  // dims (innermost first): 64 columns, rows (tokens or heads), 9 column chunks
  const cuuint64_t gq[3] = {64, cuuint64_t(s.batch) * kHeads, 9};
  const cuuint64_t sq[2] = {cuuint64_t(kDk) * 2, 128};
  const cuuint64_t gk[3] = {64, cuuint64_t(s.num_pages) * s.page_size, 9};
  const cuuint64_t sk[2] = {cuuint64_t(s.v_row_stride) * 2, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  for (int r = 0; r < 2; ++r) {
    const cuuint32_t nch = r == 0 ? 4 : 5;
    const cuuint32_t bq[3] = {64, kHeads, nch}, bk[3] = {64, kBlk, nch};
    if (encode_tiled(&tq[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), gq, sq, bq, es,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tiled(&tkv[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), gk, sk, bk, es,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SKD_EINVAL;
  }
  Params p;
  p.page_table = a.page_table;
  p.seqlens = a.seqlens;
  p.plan = a.plan;
  uint8_t *ws = static_cast<uint8_t *>(a.ws);
  p.err = reinterpret_cast<int32_t *>(ws);
  p.item_cnt = reinterpret_cast<int32_t *>(ws + a.wl.counters);
  p.partials = reinterpret_cast<float *>(ws + a.wl.partials);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.batch = s.batch;
  p.P = s.page_size;
  p.max_pages = s.max_pages_per_req;
  p.num_pages = s.num_pages;
  p.max_slots = int(a.wl.slots);
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.slot_floats = a.wl.slot_floats;
  p.trace = static_cast<long long *>(trace_buffer(2 * a.n_ctas));
  // stages per rank: shared memory = fixed region + Q + stages (both ranks get the same size)
  const int budget = 227 * 1024 - 1024;
  p.nst0 = std::min(kMaxSt, (budget - kOffQ - 4 * kHeads * 128) / (4 * kBlk * 128));
  p.nst1 = std::min(kMaxSt, (budget - kOffQ - 5 * kHeads * 128) / (5 * kBlk * 128));
  if (p.nst0 < 2 || p.nst1 < 2) return SKD_EUNSUPPORTED;
  const int smem0 = kOffQ + 4 * kHeads * 128 + p.nst0 * 4 * kBlk * 128;
  const int smem1 = kOffQ + 5 * kHeads * 128 + p.nst1 * 5 * kBlk * 128;
  const int smem = std::max(smem0, smem1) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return SKD_ECUDA;
    attr_set = true;
  }
  mla_decode_kernel<<<2 * a.n_ctas, kThreads, smem, a.stream>>>(tq[0], tq[1], tkv[0], tkv[1], p);
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace skd
