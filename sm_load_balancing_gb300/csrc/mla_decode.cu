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
// One worker = a 2-CTA cluster with a producer/consumer split of the math.
// TMEM holds 128 lanes x 512 fp32 columns per SM, and the 128x512 fp32 output
// accumulator alone fills it, so the two contractions live on different SMs:
//   rank 0 (scores): Q [128 heads][576] sits in its TMEM as the A operand. It
//     arrives once per segment by TMA through the KV ring (three fills ahead of
//     the segment's blocks) and each of three issuing warps copies the chunks
//     it uses into TMEM with tcgen05.cp. S = Q K^T runs with M=128 heads, N=64
//     tokens per 64-token block: each issuer accumulates a third of K=576 into
//     its own partial tile and the eight epilogue warps add the three, run the
//     online softmax (two warps per head quarter, one thread per head row and
//     column half) and stage the bf16 probabilities P, which leave for rank 1
//     as one 16 KB bulk copy per block;
//   rank 1 (values): O += P V with M=128, N=2x256, K=64 into its TMEM.
// Each rank streams the block into its own ring: rank 0 reads it from HBM,
// rank 1 a few microseconds later, mostly from L2, as its last reader. In the
// sparse (top-k) form a block is 64 listed rows: the ranks share one ring, each
// gathers part of every block with tile::gather4 and passes it to the partner's
// stage with one DSMEM bulk copy.
// The running maximum is kept per row and only moved (with an O rescale on
// rank 1) when a block's maximum exceeds it by more than 2^8, so p <= 256 and
// rescales are rare; l and O stay consistent with the same reference maximum.
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
// warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per TMEM lane quarter),
// (sparse, rank 1) warp 10 forwards its gathered part of each block to rank 0,
// warps 10-11 (rank 0) two more MMA issuers: one thread issues a tcgen05.mma
// about every 90-120 cycles whatever its size, so the 36 small score MMAs of a
// block are spread over three issuing warps
constexpr int kThreads = 384;
constexpr int kQkIssuers = 3;
constexpr int kNst = 3;        // KV ring stages
constexpr float kTau = 8.f;    // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kTraceWords = SKD_TRACE_RECORD_BYTES / 8;
constexpr int kEpiBar = 6;  // named barrier of the 8 epilogue warps of rank 0

// shared memory (offsets are the same in both ranks: multicast commits, DSMEM
// copies and stores address the partner's buffers by the local offset)
constexpr uint32_t kChunkBytes = kBlk * 128;       // 64 columns x 64 tokens, bf16, SW128
constexpr uint32_t kMainBytes = 8 * kChunkBytes;   // value columns [0, 512) of one block
constexpr uint32_t kPBytes = kHeads * kBlk * 2;    // P of one block: 128 rows x 128 B
constexpr uint32_t kQuarterP = kPBytes / 4;        // the 32 rows of one epilogue warp
constexpr uint32_t kQChunkBytes = kHeads * 128;    // Q columns [64 c, 64 c + 64) of all heads, SW128
// sparse: rank 0 gathers value chunks [0, kGather0) and the rope chunk, rank 1
// chunks [kGather0, 8), which balances the TMA operations of the two SMs
constexpr int kGather0 = 4;
constexpr uint32_t kPart0 = kGather0 * kChunkBytes, kPart1 = (8 - kGather0) * kChunkBytes;
constexpr uint32_t kOffRing = 0;                   // [kNst][64 KB], both ranks
constexpr uint32_t kOffRope = kNst * kMainBytes;   // rank 0: [2][8 KB] columns [512, 576)
constexpr uint32_t kOffStage = kOffRope + 2 * kChunkBytes;  // rank 0: P staging [4 warps][4 KB]
constexpr uint32_t kOffP = kNst * kMainBytes;      // rank 1: P [2][128 rows][64 tok] bf16, SW128
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;  // mbarriers
constexpr int kNumBar = 28;
// per (P buffer, warp): 32 rescale factors + a flag word, padded to 144 bytes
// (rank 0 stages its copy in the slots of P buffer 0)
constexpr uint32_t kFaBytes = 144;
constexpr uint32_t kOffFa = kOffBar + kNumBar * 8;
constexpr uint32_t kOffStats = kOffFa + 8 * kFaBytes;  // rank 1: m, l, lf [3][128] fp32
constexpr uint32_t kOffMisc = kOffStats + 3 * kHeads * 4;
// misc words: 0 tmem base, 1 abort, 2 merge decision, 3 blocks issued by the producer,
// 4 (sparse, rank 1) per stage: bit s parity of the gather phases issued, bit 8+s any issued
constexpr uint32_t kSmemBytes = kOffMisc + 64;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffStage + 4 * kQuarterP <= kOffBar, "P staging overlaps the barriers");
static_assert(kOffFa % 16 == 0 && kFaBytes % 16 == 0, "bulk copies need 16-byte alignment");

// TMEM columns
constexpr uint32_t kTQ = 0;                     // rank 0: Q, 288 columns (2 bf16 per column)
constexpr uint32_t kTS = 320;                   // rank 0: 3 partial score tiles (one per issuer), 64 columns each
constexpr uint32_t kTO = 0;                     // rank 1: O, 512 columns

enum {
  B_KVF = 0,            // [kNst] block landed (rank 0: 72 KB, rank 1: 64 KB)
  B_KVE = kNst,         // [kNst] stage free (rank 0: QK done, rank 1: PV done)
  B_RE0 = 2 * kNst,     // [2] rank 0: rope slot free (QK done)
  B_Q0 = B_RE0 + 2,     // rank 1: rank 0 has its first Q (1 remote arrival, once)
  B_SF0, B_SF1,         // rank 0: score tiles complete (3 issuers; B_SF1 unused)
  B_SE0, B_SE1,         // rank 0: score tiles read out (8 epilogue warps; B_SE1 unused)
  B_PF0, B_PF1,         // rank 1: P, factors and flags of the block landed (2 bulk copies)
  B_PVD0, B_PVD1,       // both: PV of the block that used P buffer 0/1 complete
  B_OR0, B_OR1,         // rank 1: O rescaled / V tail zeroed, PV may run (4)
  B_STF,                // rank 1: segment statistics landed (4 remote)
  B_STE,                // rank 0: statistics buffer free (4 remote)
  B_KVH,                // [kNst] sparse: this CTA's own gathers of a fill landed
  B_FIN = B_KVH + kNst,  // MMA drain before TMEM release
  B_COUNT
};
static_assert(B_COUNT <= kNumBar, "barrier count");

struct Params {
  const int32_t *page_table;
  const int32_t *seqlens;
  const int32_t *plan;
  int32_t *err;
  int32_t *item_cnt;
  float *partials;
  __nv_bfloat16 *out;
  float *lse;
  int batch, P, max_pages, num_pages, max_slots;
  float scale_log2;
  int64_t slot_floats;
  long long *trace;
  int defer;  // 1: splits write their partial states and a combine kernel merges them
  // sparse (top-k) attention: request b attends to the cache positions
  // topk[b * topk_stride + i], i < topk_len[b] (the plan splits those lists);
  // topk == nullptr: every position of the cache (dense)
  const int32_t *topk;
  const int32_t *topk_len;
  int topk_stride;
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
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// the same without release semantics (the data follows through the async proxy)
__device__ __forceinline__ void arrive_expect_tx_remote_relaxed(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
               "r"(bytes)
               : "memory");
}
// copy `bytes` of this CTA's shared memory to the partner's (cluster address),
// counted on the partner's barrier `bar_cluster`
__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
// four listed rows x one 64-column box of a 2-D map (one row high) into 512
// consecutive bytes of shared memory, swizzled like a 4-row slice of a tile
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *m, uint32_t bar, int col, int r0, int r1,
                                            int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// fp32 store that asks L2 to keep the line (partials are read again at the kernel's end)
__device__ __forceinline__ void st_keep(float *p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled store shared -> global (bulk group)
__device__ __forceinline__ void tma_store2(const CUtensorMap *m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
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
// D (TMEM) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
// D (TMEM) (+)= A (TMEM: lane = row, column c = elements 2c, 2c+1) * B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
// TMEM (128 lanes x 8 columns from taddr) <- 128 rows x 32 bytes of shared
// memory given by an operand descriptor; ordered before later MMAs of the same thread
__device__ __forceinline__ void tmem_cp128(uint32_t taddr, uint64_t sd) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sd) : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// arrive on the barrier at the same offset in every CTA of `mask`
__device__ __forceinline__ void umma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns per warp (lane = TMEM lane of the warp's quarter)
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
// the same load without its wait, and a wait that the 32 results depend on
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
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

// trace words 2..11: cycles spent waiting, per barrier kind (lane 0 of each waiting warp)
__device__ __forceinline__ int trace_word(int i) {
  return i < B_KVE ? 2 : i < B_Q0 ? 3 : i == B_Q0 ? 4 : i <= B_SF1 ? 5 : i <= B_SE1 ? 6 : i <= B_PF1 ? 7
       : i <= B_PVD1 ? 8 : i <= B_OR1 ? 9 : i == B_STF ? 10 : 11;
}

struct Ctx {
  uint32_t sbase, peer;  // own shared base; peer rank
  volatile int *abort;
  int32_t *err;
  long long *tr;  // per-CTA trace record or null
  __device__ uint32_t bar(int i) const { return sbase + kOffBar + 8u * i; }
  __device__ uint32_t peer_addr(uint32_t local) const { return mapa(local, peer); }
  // a ring fill has landed: its barrier, and with the shared ring (sparse)
  // also this CTA's own part of it (parity of KVH's phase: hpar)
  __device__ bool wait_fill(int s, uint32_t parity, bool shared_ring, uint32_t hpar) const {
    return wait(B_KVF + s, parity) && (!shared_ring || wait(B_KVH + s, hpar));
  }
  // bounded wait with cluster-scope acquire; on timeout flag both ranks
  __device__ bool wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    const long long t0 = clock64();
    if (try_wait_cluster(b, parity)) {
      if (tr && (threadIdx.x & 31) == 0)
        atomicAdd(reinterpret_cast<unsigned long long *>(tr + trace_word(i)), (unsigned long long)(clock64() - t0));
      return true;
    }
    uint32_t n = 0;
    bool ok = true;
    while (!try_wait_cluster(b, parity)) {
      if ((++n & 255u) == 0) {
        if (*abort) {
          ok = false;
          break;
        }
        if (clock64() - t0 > kWaitCycles) {
          *abort = 1;
          st_cluster_u32(peer_addr(sbase + kOffMisc + 4), 1u);
          atomicOr(err, SKD_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    if (tr && (threadIdx.x & 31) == 0)
      atomicAdd(reinterpret_cast<unsigned long long *>(tr + trace_word(i)), (unsigned long long)(clock64() - t0));
    return ok;
  }
};

// number of 64-token blocks touched by the token range [tb, te)
__device__ __forceinline__ int num_blocks(int tb, int te) { return (te + kBlk - 1) / kBlk - tb / kBlk; }

// kSparse: the top-k form (blocks of listed rows, gathered); a template
// parameter so that the dense kernel carries none of its code
template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmain, const __grid_constant__ CUtensorMap trope,
                      const __grid_constant__ CUtensorMap tpart, const __grid_constant__ CUtensorMap tout,
                      const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tg,
                      const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // with programmatic dependent launch this grid may start before the previous
  // kernel of the stream (e.g. the device planner) has finished: wait for it
  // before reading any input
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  Ctx cx;
  cx.sbase = ptx::smem_u32(smem);
  // the 128-byte swizzle needs 1024-byte aligned tiles; the dynamic window
  // starts aligned when the kernel declares no static shared memory
  if (cx.sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, SKD_DEVERR_PLAN);
    return;  // same offset in both ranks
  }
  const PlanOffsets off = plan_offsets(p.batch, 1, nworkers);
  const int seg_lo = plan[off.cta_off + worker], seg_hi = plan[off.cta_off + worker + 1];
  const int4 *segs = reinterpret_cast<const int4 *>(plan + off.segs);

  cx.peer = rank ^ 1u;
  cx.abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  cx.err = p.err;
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc);

  constexpr bool sparse = kSparse;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNst; ++s) {
      ptx::mbar_init(cx.bar(B_KVF + s), 1);
      // sparse: one ring shared by the pair (every block lands in both CTAs);
      // rank 0's 3 score issuers and rank 1's PV issuer release a fill in
      // both CTAs, and rank 1's forwarding warp in its own as well
      ptx::mbar_init(cx.bar(B_KVE + s), sparse ? kQkIssuers + 1 + rank : rank == 0 ? kQkIssuers : 1);
    }
    ptx::mbar_init(cx.bar(B_RE0), 1);
    ptx::mbar_init(cx.bar(B_RE0 + 1), 1);
    ptx::mbar_init(cx.bar(B_Q0), 1);
    ptx::mbar_init(cx.bar(B_SF0), kQkIssuers);
    ptx::mbar_init(cx.bar(B_SF1), 1);
    ptx::mbar_init(cx.bar(B_SE0), 8);
    ptx::mbar_init(cx.bar(B_SE1), 8);
    ptx::mbar_init(cx.bar(B_PF0), 1);
    ptx::mbar_init(cx.bar(B_PF1), 1);
    ptx::mbar_init(cx.bar(B_PVD0), 1);
    ptx::mbar_init(cx.bar(B_PVD1), 1);
    ptx::mbar_init(cx.bar(B_OR0), 8);
    ptx::mbar_init(cx.bar(B_OR1), 8);
    ptx::mbar_init(cx.bar(B_STF), 4);
    ptx::mbar_init(cx.bar(B_STE), 8);
    for (int s = 0; s < kNst; ++s) ptx::mbar_init(cx.bar(B_KVH + s), 1);
    ptx::mbar_init(cx.bar(B_FIN), rank == 0 ? kQkIssuers : 1);
    misc[1] = 0;
    misc[3] = 0;
    misc[4] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(cx.sbase + kOffMisc),
                 "r"(512u));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();  // barriers of both ranks initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = misc[0];

  long long *const tr = p.trace ? p.trace + int64_t(blockIdx.x) * kTraceWords : nullptr;
  cx.tr = tr;
  if (tr && threadIdx.x == 0) tr[0] = (long long)ptx::globaltimer_ns();

  const int q4 = warp & 3;                       // TMEM lane quarter of an epilogue warp
  const int hc = (warp - 2) >> 2;                // its half (score columns on rank 0, O columns on rank 1)
  const int row = q4 * 32 + lane;                // query head of an epilogue thread
  const uint32_t lane_off = uint32_t(q4 * 32) << 16;

  if (warp == 0) {
    // ============================ TMA producers ==============================
    // Each rank loads its own copy of the value columns into its own ring, so
    // a rank-0 stage is free again as soon as its score MMAs are done; rank 1
    // reads the block a few microseconds later, from L2, as its last reader.
    const uint64_t pol = rank == 0 ? policy_evict_normal() : ptx::policy_evict_first();
    int g = 0, m = 0;  // KV blocks, ring fills (on rank 0 Q takes three fills per segment)
    bool ok = true;
    for (int si = seg_lo; si < seg_hi && ok; ++si) {
      const int4 sg = segs[si];
      const int b = sg.x, tb = sg.y, te = sg.z;
      if (te <= tb) continue;
      const int32_t *ptab = p.page_table + int64_t(b) * p.max_pages;
      const int L = p.seqlens[b];
      const int len = sparse ? p.topk_len[b] : L;  // entries of the list the plan splits
      if (lane == 0 && (te > len || L > p.max_pages * p.P || (sparse && len > p.topk_stride)))
        atomicOr(p.err, SKD_DEVERR_SEQLEN);
      if (rank == 0 || sparse) {
        // the segment's Q [128 heads][576] comes through the ring ahead of its
        // blocks, as fills of chunks 0-3, 4-7 and 8 (16 KB each); the issuers
        // copy it into TMEM. With the shared ring (sparse) rank 0's Q counts as
        // its own part (KVH), and rank 1 passes the same fills with an empty
        // arrival on KVF: its KVH counts only the blocks it gathers, so that
        // the forwarding warp, which skips Q fills, can never be two phases
        // behind on a stage.
        for (int qb = 0; qb < 3 && ok; ++qb, ++m) {
          const int s = m % kNst;
          if (lane == 0) {
            ok = cx.wait(B_KVE + s, (uint32_t(m / kNst) & 1u) ^ 1u);
            if (ok) {
              const int nch = qb < 2 ? 4 : 1;
              const uint32_t qbar = cx.bar((sparse ? B_KVH : B_KVF) + s);
              if (rank == 0) {
                ptx::mbar_arrive_expect_tx(qbar, uint32_t(nch) * kQChunkBytes);
                for (int c = 0; c < nch; ++c)
                  tma3(cx.sbase + kOffRing + s * kMainBytes + c * kQChunkBytes, &tq, qbar, 0, b * kHeads, 4 * qb + c,
                       pol);
              }
              if (sparse) ptx::mbar_arrive(cx.bar(B_KVF + s));  // nothing comes from the partner
              misc[3] = uint32_t(m + 1);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      // sparse: the cache row of list entry e (row 0 past the list); each lane
      // resolves two entries of a block, one block ahead of its gather, so the
      // two dependent loads (list, page table) overlap the previous block
      const int32_t *sel = sparse ? p.topk + int64_t(b) * p.topk_stride : nullptr;
      auto resolve = [&](int e) -> int {
        if (e >= len || e >= p.topk_stride) return 0;
        int j = __ldg(sel + e);
        if (j < 0 || j >= L) {
          atomicOr(p.err, SKD_DEVERR_INDEX);
          j = 0;
        }
        int pg = j / p.P < p.max_pages ? __ldg(ptab + j / p.P) : -1;
        if (pg < 0 || pg >= p.num_pages) {
          atomicOr(p.err, SKD_DEVERR_PAGE);
          pg = 0;
          j = 0;
        }
        return pg * p.P + j % p.P;
      };
      int next_a = 0, next_b = 0;
      if (sparse) {
        const int w = (tb / kBlk) * kBlk;
        next_a = resolve(w + lane);
        next_b = resolve(w + 32 + lane);
      }
      for (int w0 = (tb / kBlk) * kBlk; w0 < te && ok; w0 += kBlk, ++g, ++m) {
        const int s = m % kNst;
        const uint32_t ph = uint32_t(m / kNst) & 1u;
        if (sparse) {
          const int ra = next_a, rb = next_b;
          if (w0 + kBlk < te) {
            next_a = resolve(w0 + kBlk + lane);
            next_b = resolve(w0 + kBlk + 32 + lane);
          }
          // the block is list entries [w0, w0 + 64): tile::gather4 TMA copies
          // bring 4 listed cache rows x 64 columns per op into the 128-byte
          // swizzled stage (16 ops per column chunk, lane c issuing chunk c).
          // The ring is shared: rank 0 gathers value chunks [0, kGather0) and
          // the rope chunk, rank 1 the other value chunks, each into its own
          // stage (barrier KVH), and each CTA passes its part to the partner's
          // stage (the partner's KVF) with one bulk copy, so each SM's TMA unit
          // issues a similar share of the block's gather operations (plain ones:
          // a multicast gather costs the issuing SM about twice as much).
          // Entries past the list read row 0 of the cache: their scores are
          // masked and rank 1 zeroes their V rows.
          if (lane == 0) {
            ok = (rank == 0 || g != 1 || cx.wait(B_Q0, 0)) && cx.wait(B_KVE + s, ph ^ 1u) &&
                 (rank == 1 || cx.wait(B_RE0 + (g & 1), uint32_t((g >> 1) & 1) ^ 1u));
            if (ok) {
              ptx::mbar_arrive_expect_tx(cx.bar(B_KVH + s), rank == 0 ? kPart0 + kChunkBytes : kPart1);
              ptx::mbar_arrive_expect_tx(cx.bar(B_KVF + s), rank == 0 ? kPart1 : kPart0);
              misc[4] = (misc[4] ^ (1u << s)) | (256u << s);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          const uint32_t ring = cx.sbase + kOffRing + s * kMainBytes;
          const uint32_t rope = cx.sbase + kOffRope + (g & 1) * kChunkBytes;
          // this rank's chunks: lane c issues chunk c (lane 8: rope, rank 0)
          const bool mine = rank == 0 ? (lane < kGather0 || lane == 8) : (lane >= kGather0 && lane < 8);
#pragma unroll 1
          for (int i = 0; i < kBlk / 4; ++i) {
            int r4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int t = 4 * i + u;
              r4[u] = __shfl_sync(0xffffffffu, t < 32 ? ra : rb, t & 31);
            }
            if (mine)
              tma_gather4((lane < 8 ? ring + lane * kChunkBytes : rope) + uint32_t(i) * 512, &tg, cx.bar(B_KVH + s),
                          lane * 64, r4[0], r4[1], r4[2], r4[3]);
          }
          if (lane == 0) misc[3] = uint32_t(m + 1);
          continue;
        }
        if (lane == 0) {
          const int j = w0 / p.P;
          int pg = j < p.max_pages ? __ldg(ptab + j) : -1;
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.err, SKD_DEVERR_PAGE);
            pg = 0;
          }
          // rank 1 loads its second block only once rank 0 has its first Q,
          // which would otherwise queue behind the whole value ring of every worker
          ok = (rank == 0 || g != 1 || cx.wait(B_Q0, 0)) && cx.wait(B_KVE + s, ph ^ 1u) &&
               (rank == 1 || cx.wait(B_RE0 + (g & 1), uint32_t((g >> 1) & 1) ^ 1u));
          if (ok) {
            const int rowk = pg * p.P + (w0 % p.P);
            ptx::mbar_arrive_expect_tx(cx.bar(B_KVF + s), rank == 0 ? kMainBytes + kChunkBytes : kMainBytes);
            tma3(cx.sbase + kOffRing + s * kMainBytes, &tmain, cx.bar(B_KVF + s), 0, rowk, 0, pol);
            if (rank == 0)
              tma3(cx.sbase + kOffRope + (g & 1) * kChunkBytes, &trope, cx.bar(B_KVF + s), 0, rowk, 8, pol);
            misc[3] = uint32_t(m + 1);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
  } else if (warp == 1 || (rank == 0 && warp >= 10)) {
    // ============================ MMA issuers ================================
    if (lane == 0) {
      const uint32_t part_src = cx.sbase + kOffRing;  // rank 0's value part: chunks [0, kGather0) of a stage
      int g = 0;
      bool ok = true;
      if (rank == 0) {
        // issuer qi accumulates latent chunks [3 qi, 3 qi + 3) into its own
        // partial score tile; the epilogue adds the three tiles
        const int qi = warp == 1 ? 0 : warp - 9;
        constexpr uint32_t id_qk = idesc(kHeads, kBlk, 0);
        const uint32_t dS = tmem + kTS + 64 * qi;
        int m = 0;  // ring fills, as counted by the producer
        for (int si = seg_lo; si < seg_hi && ok; ++si) {
          const int4 sg = segs[si];
          if (sg.z <= sg.y) continue;
          const int nb = num_blocks(sg.y, sg.z);
          // Q of the segment: this issuer copies the three chunks its MMAs use
          // from the ring into TMEM, once the score MMAs of the previous block
          // (the last readers of those columns) are complete
          if (g > 0) ok = cx.wait(B_SF0, uint32_t((g - 1) & 1));
          for (int qb = 0; qb < 3 && ok; ++qb) {
            const uint32_t par = uint32_t((m + qb) / kNst) & 1u;
            ok = cx.wait_fill((m + qb) % kNst, par, sparse, par);
          }
          if (!ok) break;
          tc_fence_after();
          if (g == 0 && qi == 0) arrive_remote(cx.peer_addr(cx.bar(B_Q0)));
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {
            const int c = 3 * qi + cc, f = m + c / 4;  // chunk c sits in fill f
            const uint32_t src = cx.sbase + kOffRing + uint32_t(f % kNst) * kMainBytes + uint32_t(c % 4) * kQChunkBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tmem_cp128(tmem + kTQ + c * 32 + kk * 8, sdesc(src + kk * 32, 16, 1024));
          }
          for (int qb = 0; qb < 3; ++qb) {
            if (sparse)
              umma_commit_mc(cx.bar(B_KVE + (m + qb) % kNst), 0x3);
            else
              umma_commit(cx.bar(B_KVE + (m + qb) % kNst));
          }
          m += 3;
          for (int j = 0; j < nb && ok; ++j, ++g, ++m) {
            const int s = m % kNst;
            if (sparse && qi == 0) {
              // issuer 0 passes rank 0's gathered value part to rank 1 as soon
              // as it has landed (it waits for this stage anyway)
              if (!cx.wait(B_KVH + s, uint32_t(m / kNst) & 1u)) {
                ok = false;
                break;
              }
              const uint32_t src = part_src + uint32_t(s) * kMainBytes;
              bulk_s2s(cx.peer_addr(src), src, kPart0, cx.peer_addr(cx.bar(B_KVF + s)));
              bulk_commit();
            }
            const uint32_t par = uint32_t(m / kNst) & 1u;
            if (!cx.wait_fill(s, par, sparse, par) || !cx.wait(B_SE0, uint32_t(g & 1) ^ 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t ring = cx.sbase + kOffRing + s * kMainBytes;
            const uint32_t rope = cx.sbase + kOffRope + (g & 1) * kChunkBytes;
#pragma unroll
            for (int cc = 0; cc < 3; ++cc) {
              const int c = 3 * qi + cc;
              const uint32_t bc = c < 8 ? ring + c * kChunkBytes : rope;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ts(dS, tmem + kTQ + c * 32 + kk * 8, sdesc(bc + kk * 32, 16, 1024), id_qk, (cc | kk) != 0);
            }
            umma_commit(cx.bar(B_SF0));
            if (sparse && qi == 0) bulk_wait_read0();  // the copy to rank 1 has read the stage
            if (sparse)
              umma_commit_mc(cx.bar(B_KVE + s), 0x3);  // the stage is shared with rank 1
            else
              umma_commit(cx.bar(B_KVE + s));
            if (qi == 2) umma_commit(cx.bar(B_RE0 + (g & 1)));
          }
        }
      } else {
        constexpr uint32_t id_pv = idesc(kHeads, 256, 1);
        int m = 0;  // ring fills: the blocks, and with the shared ring (sparse) rank 0's Q fills too
        uint32_t hp = 0;  // per stage, parity of this CTA's next gather phase (KVH counts blocks only)
        for (int si = seg_lo; si < seg_hi && ok; ++si) {
          const int4 sg = segs[si];
          if (sg.z <= sg.y) continue;
          const int nb = num_blocks(sg.y, sg.z);
          if (sparse) {
            // the segment's three Q fills pass through this CTA's ring too: release them
            for (int qb = 0; qb < 3 && ok; ++qb, ++m) {
              ok = cx.wait(B_KVF + m % kNst, uint32_t(m / kNst) & 1u);
              if (ok) umma_commit_mc(cx.bar(B_KVE + m % kNst), 0x3);
            }
          }
          for (int j = 0; j < nb && ok; ++j, ++g, ++m) {
            const int s = m % kNst, pb = g & 1;
            if (!cx.wait_fill(s, uint32_t(m / kNst) & 1u, sparse, (hp >> s) & 1u) ||
                !cx.wait(B_OR0 + pb, uint32_t((g >> 1) & 1))) {
              ok = false;
              break;
            }
            hp ^= 1u << s;
            tc_fence_after();
            const uint32_t ring = cx.sbase + kOffRing + s * kMainBytes;
            const uint32_t pbuf = cx.sbase + kOffP + pb * kPBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc(pbuf + kk * 32, 16, 1024);
#pragma unroll
              for (int h = 0; h < 2; ++h)
                umma_ss(tmem + kTO + h * 256, a, sdesc(ring + h * 4 * kChunkBytes + kk * (16 * 128), 8192, 1024),
                        id_pv, (j > 0 || kk > 0) ? 1u : 0u);
            }
            if (sparse)
              umma_commit_mc(cx.bar(B_KVE + s), 0x3);  // the stage is shared with rank 0
            else
              umma_commit(cx.bar(B_KVE + s));
            umma_commit_mc(cx.bar(B_PVD0 + pb), 0x3);  // P buffer free (rank 0), O ready (rank 1)
          }
        }
      }
      if (sparse) bulk_wait0();  // rank 0 issuer 0's copies to rank 1 have read their stages
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(cx.bar(B_FIN));
      ptx::mbar_wait(cx.bar(B_FIN), 0, nullptr, kWaitCycles);
    }
  } else if (rank == 0 && warp >= 2 && warp < 10) {
    // ====================== rank 0 epilogue: online softmax ====================
    // Warps w and w+4 share the 32 head rows of one TMEM lane quarter; warp
    // half hc handles score columns [32 hc, 32 hc + 32) of every block. The
    // two halves exchange their row maxima through shared memory, so both
    // derive the same reference maximum, and keep separate partial sums.
    float *xm = reinterpret_cast<float *>(smem + kOffStats);  // [2 halves][128 rows]
    const int pair_bar = 2 + q4;
    int g = 0, stn = 0;
    bool ok = true;
    for (int si = seg_lo; si < seg_hi; ++si) {
      const int4 sg = segs[si];
      const int tb = sg.y, te = sg.z;
      if (te <= tb) continue;
      const int nb = num_blocks(tb, te);
      float mref = -INFINITY, l = 0.f, lf = 0.f;  // l, lf: this half's sums
      const uint32_t stage = cx.sbase + kOffStage + uint32_t(q4) * kQuarterP;  // the quarter's P rows
      const uint32_t fstage = cx.sbase + kOffFa + uint32_t(q4) * kFaBytes;    // its factors + flag
      for (int j = 0; j < nb; ++j, ++g) {
        const int w0 = (tb / kBlk) * kBlk + j * kBlk;
        const int pb = g & 1;
        float s[32];
        ok = ok && cx.wait(B_SF0, uint32_t(g & 1));
        tc_fence_after();
        {
          // the three partial tiles, loaded together and waited for once
          uint32_t r0[32], r1[32], r2[32];
          const uint32_t tS = tmem + kTS + lane_off + 32 * hc;
          tmem_ld32_async(tS, r0);
          tmem_ld32_async(tS + 64, r1);
          tmem_ld32_async(tS + 128, r2);
          tmem_wait_ld(r0);
          tmem_wait_ld(r1);
          tmem_wait_ld(r2);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = (__uint_as_float(r0[c]) + __uint_as_float(r1[c])) + __uint_as_float(r2[c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cx.bar(B_SE0));
        // tokens outside [tb, te) do not take part (the block may start
        // before the segment or run past it); the check is warp-uniform
        const int lo = tb - w0 - 32 * hc, hi = te - w0 - 32 * hc;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (lo <= 0 && hi >= 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], s[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < lo || c >= hi) s[c] = -INFINITY;
            m4[c & 3] = fmaxf(m4[c & 3], s[c]);
          }
        }
        // the staging tile is free once the previous block's copies have read it
        if (warp == 2 && lane == 0) bulk_wait_read0();
        xm[hc * kHeads + row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        ptx::named_bar(kEpiBar, 256);  // maxima exchanged; the staging tile is free for every warp
        // scores are scaled into log2 units on the fly: the scale is positive,
        // so the maximum of the scaled scores is the scaled maximum
        const float mx = fmaxf(xm[row], xm[kHeads + row]) * p.scale_log2;
        float a = 1.f;
        if (j == 0) {
          mref = mx;
        } else if (mx > mref + kTau) {
          a = ex2(mref - mx);
          mref = mx;
          l *= a;
          lf *= a;
        }
        uint32_t pk[16];
        float ps2[2] = {0.f, 0.f}, pf2[2] = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float e0 = ex2(fmaf(s[c], p.scale_log2, -mref)), e1 = ex2(fmaf(s[c + 1], p.scale_log2, -mref));
          pf2[(c >> 1) & 1] += e0 + e1;
          pk[c / 2] = ptx::pack_bf16(e0, e1);
          const float2 f = ptx::unpack_bf16(pk[c / 2]);
          ps2[(c >> 1) & 1] += f.x + f.y;
        }
        l += ps2[0] + ps2[1];
        lf += pf2[0] + pf2[1];
        // stage this half of the quarter's 32 P rows (the 128-byte swizzle
        // depends only on row & 7, so the 4 KB tile lands in rank 1 with its
        // final layout); half 0 also stages the rescale factors and flag
        {
          const uint32_t srow = stage + uint32_t(lane) * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = 4 * hc + k;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + uint32_t((c ^ (row & 7)) << 4)),
                         "r"(pk[4 * k]), "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                         : "memory");
          }
          if (hc == 0) {
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(fstage + uint32_t(lane) * 4), "f"(a) : "memory");
            const uint32_t any = __any_sync(0xffffffffu, a != 1.f) ? 1u : 0u;
            if (lane == 0) asm volatile("st.shared.u32 [%0], %1;" ::"r"(fstage + 128), "r"(any) : "memory");
          }
        }
        ptx::fence_proxy_async_smem();  // staged bytes are read by the bulk copy (async proxy)
        ptx::named_bar(kEpiBar, 256);
        // one bulk copy of the whole 16 KB tile (and one of the four quarters'
        // factors) into P buffer pb of rank 1 once PV(g-2), its previous
        // reader, is done: a few large copies keep the hand-over short
        if (warp == 2 && lane == 0) {
          ok = ok && cx.wait(B_PVD0 + pb, uint32_t(((g >> 1) & 1) ^ 1));
          const uint32_t pf = cx.peer_addr(cx.bar(B_PF0 + pb));
          arrive_expect_tx_remote_relaxed(pf, 4 * (kQuarterP + kFaBytes));
          bulk_s2s(cx.peer_addr(cx.sbase + kOffP + uint32_t(pb) * kPBytes), cx.sbase + kOffStage, 4 * kQuarterP, pf);
          bulk_s2s(cx.peer_addr(cx.sbase + kOffFa + uint32_t(pb * 4) * kFaBytes), cx.sbase + kOffFa, 4 * kFaBytes,
                   pf);
          bulk_commit();
        }
      }
      // segment end: the two halves' sums, then the row statistics to rank 1
      if (hc == 1) {
        xm[row] = l;
        xm[kHeads + row] = lf;
      }
      ptx::named_bar(pair_bar, 64);
      if (hc == 0) {
        l += xm[row];
        lf += xm[kHeads + row];
        ok = ok && cx.wait(B_STE, uint32_t(stn & 1) ^ 1u);
        const uint32_t st = cx.peer_addr(cx.sbase + kOffStats + uint32_t(row) * 4);
        st_cluster_f32(st, mref);
        st_cluster_f32(st + kHeads * 4, l);
        st_cluster_f32(st + 2 * kHeads * 4, lf);
        __syncwarp();
        if (lane == 0) arrive_remote(cx.peer_addr(cx.bar(B_STF)));
      }
      ++stn;
      ptx::named_bar(pair_bar, 64);  // xm is free for the next segment
    }
    if (warp == 2 && lane == 0) bulk_wait_read0();
    (void)ok;
  } else if (rank == 1 && warp >= 2 && warp < 10) {
    // ================= rank 1 epilogue: O rescale, tails, output ================
    // Warp half hc owns O columns [256 hc, 256 hc + 256) of its quarter's rows.
    const volatile float *stats = reinterpret_cast<const volatile float *>(smem + kOffStats);
    volatile int *decision = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    const uint32_t tOh = tmem + kTO + lane_off + 256 * hc;  // this thread's row, this half's columns
    const int col0 = 256 * hc;
    int g = 0, m = 0, stn = 0;  // blocks, ring fills (the shared ring also carries Q fills)
    uint32_t hp = 0;            // per stage, parity of this CTA's next gather phase (sparse)
    bool ok = true;
    for (int si = seg_lo; si < seg_hi; ++si) {
      const int4 sg = segs[si];
      const int b = sg.x, tb = sg.y, te = sg.z, wslot = sg.w;
      const int64_t orow = int64_t(b) * kHeads + row;
      if (te <= tb) {  // empty request
        uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + col0);
        for (int c = 0; c < 256 / 8; ++c) o4[c] = make_uint4(0, 0, 0, 0);
        if (hc == 0) p.lse[orow] = -INFINITY;
        continue;
      }
      const int L = sparse ? p.topk_len[b] : p.seqlens[b];  // entries of the list (positions when dense)
      const int nb = num_blocks(tb, te);
      if (sparse) m += 3;
      for (int j = 0; j < nb; ++j, ++g, ++m) {
        const int w0 = (tb / kBlk) * kBlk + j * kBlk;
        const int pb = g & 1, s = m % kNst;
        ok = ok && cx.wait(B_PF0 + pb, uint32_t((g >> 1) & 1));
        const volatile uint32_t *fa =
            reinterpret_cast<const volatile uint32_t *>(smem + kOffFa + (pb * 4 + q4) * kFaBytes);
        const uint32_t flag = fa[32];
        if (flag && j > 0) {
          // the maximum of some of this quarter's rows moved: scale their O
          // columns (after PV(g-1); PV(g) waits for this warp's arrival below)
          ok = ok && cx.wait(B_PVD0 + ((g - 1) & 1), uint32_t(((g - 1) >> 1) & 1));
          tc_fence_after();
          const float a = __uint_as_float(fa[lane]);
          float v[32];
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            tmem_ld32(tOh + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= a;
            tmem_st32(tOh + c, reinterpret_cast<const uint32_t *>(v));
          }
        }
        if (w0 + kBlk > L) {
          // V rows of the block past the end of the request hold arbitrary
          // bytes (0 * NaN would poison O): zero them in this rank's copy
          // (with the shared ring this warp may be more fills ahead of the PV
          // issuer than the ring is deep, because rank 0's Q fills sit between
          // blocks: first wait until the stage's previous fill was released by
          // every consumer, so that the parity test below can only be passed
          // by this block's fill)
          if (sparse && m >= kNst) ok = ok && cx.wait(B_KVE + s, uint32_t((m - kNst) / kNst) & 1u);
          ok = ok && cx.wait_fill(s, uint32_t(m / kNst) & 1u, sparse, (hp >> s) & 1u);
          const int t_lo = max(0, min(kBlk, L - w0));
          const int nrow = kBlk - t_lo;
          uint8_t *stg = smem + kOffRing + uint32_t(s) * kMainBytes;
          const int pieces = 8 * nrow * 8;
          for (int i = threadIdx.x - 64; i < pieces; i += 256) {
            const int c = i / (nrow * 8), rest = i - c * (nrow * 8);
            *reinterpret_cast<int4 *>(stg + c * kChunkBytes + (t_lo + (rest >> 3)) * 128 + (rest & 7) * 16) =
                make_int4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();  // zeros are read by the tensor core (async proxy)
        }
        hp ^= 1u << s;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cx.bar(B_OR0 + pb));
      }
      // ---- segment end: row statistics from rank 0, last PV, then output ----
      ok = ok && cx.wait(B_STF, uint32_t(stn & 1));
      const float mref = stats[row], l = stats[kHeads + row], lf = stats[2 * kHeads + row];
      __syncwarp();
      if (lane == 0) arrive_remote(cx.peer_addr(cx.bar(B_STE)));
      ++stn;
      ok = ok && cx.wait(B_PVD0 + ((g - 1) & 1), uint32_t(((g - 1) >> 1) & 1));
      tc_fence_after();
      if (wslot < 0) {
        const float inv = 1.f / l;
        float v[32];
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          tmem_ld32(tOh + c, v);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) pk[i / 2] = ptx::pack_bf16(v[i] * inv, v[i + 1] * inv);
          uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + col0 + c);
#pragma unroll
          for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        if (hc == 0) p.lse[orow] = (mref + log2f(lf)) * kLn2;
      } else {
        // ---- split: publish the partial, the last split merges ----
        const int nsp = plan[off.nsplit + b], s0 = plan[off.slot0 + b];
        ptx::named_bar(1, 256);  // previous use of the decision word is over
        if (threadIdx.x == 64)
          *decision = (!p.defer && !*cx.abort && ld_acquire_gpu(p.item_cnt + b) == nsp - 1) ? 1 : 0;
        ptx::named_bar(1, 256);
        // all other splits already published: merge from TMEM without writing this one
        const bool own_tmem = *decision != 0;
        bool last = own_tmem;
        if (!own_tmem) {
          // partial O is stored transposed, [512 columns][128 rows]: each warp
          // store is one 128-byte line (the 32 rows of the warp, one column)
          float *ps = p.partials + int64_t(wslot) * p.slot_floats;
          const uint64_t keep = ptx::policy_evict_last();
          float v[32];
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            tmem_ld32(tOh + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) st_keep(ps + (col0 + c + i) * kHeads + row, v[i], keep);
          }
          if (hc == 0) {
            st_keep(ps + kHeads * kDv + row, mref, keep);
            st_keep(ps + kHeads * kDv + kHeads + row, l, keep);
            st_keep(ps + kHeads * kDv + 2 * kHeads + row, lf, keep);
          }
          ptx::named_bar(1, 256);
          if (threadIdx.x == 64) {
            int lst = 0;
            if (!*cx.abort && !p.defer) {
              __threadfence();
              lst = ptx::atom_add_acq_rel_gpu(p.item_cnt + b, 1) == nsp - 1 ? 1 : 0;
            }
            *decision = lst;
          }
          ptx::named_bar(1, 256);
          last = *decision != 0;
        }
        if (last) {
          if (threadIdx.x == 64) p.item_cnt[b] = 0;  // ready for the next launch
          // merge all splits of this row in slot order (same arithmetic whichever split merges);
          // up to kU splits' statistics are loaded in one batch
          constexpr int kU = 8;
          float mv[kU], lv[kU], lfv[kU];
          float Mx = -INFINITY;
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            mv[u] = -INFINITY;
            lv[u] = lfv[u] = 0.f;
            if (u < nsp) {
              if (own_tmem && s0 + u == wslot) {
                mv[u] = mref;
                lv[u] = l;
                lfv[u] = lf;
              } else {
                const float *ps = p.partials + int64_t(s0 + u) * p.slot_floats + kHeads * kDv;
                mv[u] = __ldcg(ps + row);
                lv[u] = __ldcg(ps + kHeads + row);
                lfv[u] = __ldcg(ps + 2 * kHeads + row);
              }
            }
            Mx = fmaxf(Mx, mv[u]);
          }
          for (int sp = kU; sp < nsp; ++sp)
            Mx = fmaxf(Mx, (own_tmem && s0 + sp == wslot)
                               ? mref
                               : __ldcg(p.partials + int64_t(s0 + sp) * p.slot_floats + kHeads * kDv + row));
          const float Mu = Mx == -INFINITY ? 0.f : Mx;
          float lam = 0.f, lamf = 0.f;
#pragma unroll
          for (int u = 0; u < kU; ++u)
            if (u < nsp) {
              const float f = exp2f(mv[u] - Mu);
              lam += lv[u] * f;
              lamf += lfv[u] * f;
            }
          for (int sp = kU; sp < nsp; ++sp) {
            float ms, ls, lfs;
            if (own_tmem && s0 + sp == wslot) {
              ms = mref;
              ls = l;
              lfs = lf;
            } else {
              const float *ps = p.partials + int64_t(s0 + sp) * p.slot_floats + kHeads * kDv;
              ms = __ldcg(ps + row);
              ls = __ldcg(ps + kHeads + row);
              lfs = __ldcg(ps + 2 * kHeads + row);
            }
            const float f = exp2f(ms - Mu);
            lam += ls * f;
            lamf += lfs * f;
          }
          const float inv = 1.f / lam;
          const int own = wslot - s0;
          if (si == seg_hi - 1 && nsp <= 63) {
            // Fast path (the merge of a worker's last segment, the usual case:
            // the other splits finished long before): the KV ring is idle, so
            // the other splits' partial O stream into it by TMA, per warp 4
            // slots of 32 rows x 32 columns; this split's O comes from TMEM, and
            // the bf16 result leaves through two 4 KB staging tiles by TMA.
            constexpr int kMs = 4;
            const int n_o = nsp - 1, total = 8 * n_o;  // items: (32-column chunk, other split)
            const int wi = warp - 2;                    // 0..7
            const uint32_t mring = cx.sbase + kOffRing + uint32_t(wi) * (kMs * 4096 + 8192);
            const uint32_t ostage = mring + kMs * 4096;
            const uint32_t mbar = cx.sbase + kOffP + uint32_t(wi) * 32;  // P buffers are idle too
            float *fw = reinterpret_cast<float *>(smem + kOffP + 256);  // per-split weights [split][row]
            const uint64_t pol = ptx::policy_evict_first();
            if (hc == 0) {
#pragma unroll
              for (int u = 0; u < kU; ++u)
                if (u < nsp) fw[u * kHeads + row] = exp2f(mv[u] - Mu);
              for (int sp = kU; sp < nsp; ++sp)
                fw[sp * kHeads + row] = exp2f(
                    (sp == own ? mref : __ldcg(p.partials + int64_t(s0 + sp) * p.slot_floats + kHeads * kDv + row)) -
                    Mu);
            }
            if (lane == 0) {
              for (int k = 0; k < kMs; ++k) ptx::mbar_init(mbar + 8 * k, 1);
              ptx::fence_mbar_init();
            }
            ptx::named_bar(1, 256);  // weights visible to both halves
            auto issue = [&](int i) {
              const int slot = i % kMs, c = i / n_o, k = i % n_o, sp = k + (k >= own ? 1 : 0);
              ptx::mbar_arrive_expect_tx(mbar + 8 * slot, 4096);
              tma3(mring + slot * 4096, &tpart, mbar + 8 * slot, q4 * 32, col0 + c * 32, s0 + sp, pol);
            };
            int issued = 0;
            // the TMA reads partials published by other CTAs (acquired above)
            // through the async proxy
            if (lane == 0) ptx::fence_proxy_async_global();
            if (lane == 0)
              for (; issued < min(kMs, total); ++issued) issue(issued);
            int it = 0;
            bool mok = true;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {  // 32-column chunks of this half
              float acc[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
#pragma unroll 1
              for (int sp = 0; sp < nsp; ++sp) {
                float v[32];
                if (sp == own) {
                  tmem_ld32(tOh + c * 32, v);
                } else {
                  const int slot = it % kMs;
                  if (mok && !ptx::mbar_wait(mbar + 8 * slot, uint32_t(it / kMs) & 1u, cx.abort, kWaitCycles)) {
                    mok = false;
                    if (lane == 0 && !*cx.abort) {
                      *cx.abort = 1;
                      atomicOr(p.err, SKD_DEVERR_TIMEOUT);
                    }
                  }
                  // a box holds 32 columns x 32 rows (128 B per column); the
                  // 16-byte chunk k (rows 4k..4k+3) of column j sits at k ^ (j & 7)
                  const uint32_t rb = mring + slot * 4096 + uint32_t(lane & 3) * 4;
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj)
                    asm volatile("ld.shared.f32 %0, [%1];"
                                 : "=f"(v[jj])
                                 : "r"(rb + uint32_t(jj) * 128 + uint32_t((((lane >> 2) ^ (jj & 7)) << 4)))
                                 : "memory");
                  __syncwarp();  // the slot is read before it is refilled
                  if (lane == 0 && issued < total && mok) issue(issued++);
                  ++it;
                }
                const float f = fw[sp * kHeads + row];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] += v[i] * f;
              }
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) pk[i / 2] = ptx::pack_bf16(acc[i] * inv, acc[i + 1] * inv);
              // a 64-column output tile is two chunks; tile (c/2) & 1 is free
              // once the store issued two tiles ago has read it
              if ((c & 1) == 0) {
                if (lane == 0 && c >= 4) bulk_wait_read1();
                __syncwarp();
              }
              const uint32_t ot = ostage + uint32_t((c >> 1) & 1) * 4096 + uint32_t(lane) * 128;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int cc = 4 * (c & 1) + k;
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ot + uint32_t((cc ^ (lane & 7)) << 4)),
                             "r"(pk[4 * k]), "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                             : "memory");
              }
              if (c & 1) {
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store2(&tout, ostage + uint32_t((c >> 1) & 1) * 4096, col0 + (c >> 1) * 64, b * kHeads + q4 * 32);
                  bulk_commit();
                }
              }
            }
            if (lane == 0) bulk_wait0();
            // after a give-up, the loads still in flight land before the CTA leaves
            if (lane == 0)
              for (int i = it; i < issued; ++i)
                ptx::mbar_wait(mbar + 8 * (i % kMs), uint32_t(i / kMs) & 1u, nullptr, kWaitCycles);
            __syncwarp();
          } else {
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
              float acc[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
              for (int sp = 0; sp < nsp; ++sp) {
                float v[32];
                float ms;
                if (sp == own) {
                  tmem_ld32(tOh + c, v);
                  ms = mref;
                } else {
                  const float *ps = p.partials + int64_t(s0 + sp) * p.slot_floats;
#pragma unroll
                  for (int i = 0; i < 32; ++i) v[i] = __ldcg(ps + (col0 + c + i) * kHeads + row);
                  ms = __ldcg(ps + kHeads * kDv + row);
                }
                const float f = exp2f(ms - Mu);
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] += v[i] * f;
              }
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) pk[i / 2] = ptx::pack_bf16(acc[i] * inv, acc[i + 1] * inv);
              uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
          if (hc == 0) p.lse[orow] = (Mx + log2f(lamf)) * kLn2;
        }
      }
      tc_fence_before();  // O reads done before the next segment's first PV overwrites it
    }
    (void)ok;
  } else if (sparse && rank == 1 && warp == 10) {
    // ======== sparse, rank 1: pass the gathered value part (chunks [kGather0, 8)) to rank 0 ========
    // (one bulk copy per block into rank 0's stage, counted on its KVF, as
    // soon as it landed here: rank 0 needs it before P, and so before rank 1's PV).
    // This warp releases every fill of the ring here, the copied ones once the
    // copy has read them, so no barrier it waits on can run two phases ahead.
    if (lane == 0) {
      int m = 0;
      uint32_t hp = 0;  // per stage, parity of the next gather phase (KVH counts blocks only)
      bool ok = true;
      for (int si = seg_lo; si < seg_hi && ok; ++si) {
        const int4 sg = segs[si];
        if (sg.z <= sg.y) continue;
        const int nb = num_blocks(sg.y, sg.z);
        // the segment's Q fills carry nothing for rank 0: release each once the
        // stage's previous fill is released (the phase this arrival belongs to
        // has then begun; a wait on KVF could pass on the previous block's phase)
        for (int qb = 0; qb < 3 && ok; ++qb, ++m) {
          ok = cx.wait(B_KVE + m % kNst, (uint32_t(m / kNst) & 1u) ^ 1u);
          if (ok) ptx::mbar_arrive(cx.bar(B_KVE + m % kNst));
        }
        for (int j = 0; j < nb && ok; ++j, ++m) {
          const int s = m % kNst;
          ok = cx.wait(B_KVH + s, (hp >> s) & 1u);
          if (!ok) break;
          hp ^= 1u << s;
          const uint32_t src = cx.sbase + kOffRing + uint32_t(s) * kMainBytes + kPart0;
          bulk_s2s(cx.peer_addr(src), src, kPart1, cx.peer_addr(cx.bar(B_KVF + s)));
          bulk_commit();
          bulk_wait_read0();
          ptx::mbar_arrive(cx.bar(B_KVE + s));
        }
      }
      bulk_wait0();  // the copies are complete before the CTAs leave
    }
  }
  // ---- teardown: both ranks leave together (the partner may still write here) ----
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (threadIdx.x == 0 && *cx.abort) {
    // after a give-up, wait (bounded) for the copies still in flight into this CTA
    const int n = int(misc[3]);
    for (int i = max(0, n - kNst); i < n; ++i) {
      ptx::mbar_wait(cx.bar(B_KVF + i % kNst), uint32_t(i / kNst) & 1u, nullptr, kWaitCycles);
      if (sparse && rank == 0) ptx::mbar_wait(cx.bar(B_KVH + i % kNst), uint32_t(i / kNst) & 1u, nullptr, kWaitCycles);
    }
    // rank 1's KVH counts its gather phases only: wait for the last one of each stage
    const uint32_t hm = misc[4];
    for (int st = 0; st < kNst && sparse && rank == 1; ++st)
      if ((hm >> (8 + st)) & 1u) ptx::mbar_wait(cx.bar(B_KVH + st), ((hm >> st) & 1u) ^ 1u, nullptr, kWaitCycles);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u));
  }
  if (tr && threadIdx.x == 0) {
    tr[14] = seg_hi - seg_lo;
    tr[15] = ptx::smid();
    tr[1] = (long long)ptx::globaltimer_ns();
  }
}

}  // namespace

namespace {

int set_smem_attr() {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes)) !=
            cudaSuccess)
      return SKD_ECUDA;
    attr_set = true;
  }
  return SKD_OK;
}

}  // namespace

int mla_resident_workers(int *n) {
  if (set_smem_attr() != SKD_OK) return SKD_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int v = 0;
  if (cudaOccupancyMaxActiveClusters(&v, mla_decode_kernel<false>, &cfg) != cudaSuccess) return SKD_ECUDA;
  *n = v;
  return SKD_OK;
}

int launch_mla(const DecodeArgs &a) {
  const skd_shape_t &s = a.shape;
  if (s.page_size % kBlk != 0) return SKD_EUNSUPPORTED;  // 64-token blocks must not straddle pages
  // latent cache viewed as {64 columns, rows (page*P + slot), 9 column chunks}
  CUtensorMap tmain, trope, tpart, tout, tq, tg;
  const cuuint64_t gk[3] = {64, cuuint64_t(s.num_pages) * s.page_size, 9};
  const cuuint64_t sk[2] = {cuuint64_t(s.v_row_stride) * 2, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  const cuuint32_t bmain[3] = {64, kBlk, 8}, brope[3] = {64, kBlk, 1};
  if (encode_tiled(&tmain, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), gk, sk, bmain, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tiled(&trope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), gk, sk, brope, es,
                   CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return SKD_EINVAL;
  // sparse gather: the latent cache as 2-D rows {576 columns, rows}, boxes one row high x 64 columns
  {
    const cuuint64_t gg[2] = {cuuint64_t(kDk), cuuint64_t(s.num_pages) * s.page_size};
    const cuuint64_t sg[1] = {cuuint64_t(s.v_row_stride) * 2};
    const cuuint32_t bg[2] = {64, 1};
    if (encode_tiled(&tg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.k), gg, sg, bg, es,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SKD_EINVAL;
  }
  // queries [batch * 128 heads][576] viewed as {64 columns, rows, 9 column chunks}, one chunk per box
  {
    const cuuint64_t gq[3] = {64, cuuint64_t(s.batch) * kHeads, 9};
    const cuuint64_t sq[2] = {cuuint64_t(kDk) * 2, 128};
    const cuuint32_t bq[3] = {64, kHeads, 1};
    if (encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), gq, sq, bq, es,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SKD_EINVAL;
  }
  // partial-state slots (O stored transposed) viewed as {128 rows, 512 columns, slots} fp32, boxes of 32 x 32
  {
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    const cuuint64_t gp[3] = {cuuint64_t(kHeads), cuuint64_t(kDv), cuuint64_t(std::max<int64_t>(a.wl.slots, 1))};
    const cuuint64_t spb[2] = {cuuint64_t(kHeads) * 4, cuuint64_t(a.wl.slot_floats) * 4};
    const cuuint32_t bp[3] = {32, 32, 1};
    if (encode_tiled(&tpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws + a.wl.partials, gp, spb, bp, es,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SKD_EINVAL;
    // output rows {512 columns, batch*128 rows} bf16, boxes of 64 x 32
    const cuuint64_t go[2] = {cuuint64_t(kDv), cuuint64_t(s.batch) * kHeads};
    const cuuint64_t so[1] = {cuuint64_t(kDv) * 2};
    const cuuint32_t bo[2] = {64, 32};
    if (encode_tiled(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, go, so, bo, es,
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
  p.defer = a.defer_merge ? 1 : 0;
  p.topk = a.topk;
  p.topk_len = a.topk_len;
  p.topk_stride = a.topk_stride;

  if (set_smem_attr() != SKD_OK) return SKD_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = p.topk ? mla_decode_kernel<true> : mla_decode_kernel<false>;
  if (cudaLaunchKernelEx(&cfg, kern, tmain, trope, tpart, tout, tq, tg, p) != cudaSuccess) return SKD_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

// The comparator's second kernel: one CTA per request, thread (row, half)
// merges one head row's 256 value columns over all splits in split order
// (partial O is stored transposed, so consecutive rows are consecutive words).
__global__ void __launch_bounds__(256, 1) mla_combine_kernel(const Params p, int n_workers) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, row = threadIdx.x & 127, col0 = (threadIdx.x >> 7) * 256;
  const PlanOffsets off = plan_offsets(p.batch, 1, n_workers);
  const int nsp = p.plan[off.nsplit + b], s0 = p.plan[off.slot0 + b];
  if (nsp < 2) return;
  float Mx = -INFINITY;
  for (int sp = 0; sp < nsp; ++sp)
    Mx = fmaxf(Mx, __ldcg(p.partials + int64_t(s0 + sp) * p.slot_floats + kHeads * kDv + row));
  const float Mu = Mx == -INFINITY ? 0.f : Mx;
  float lam = 0.f, lamf = 0.f;
  for (int sp = 0; sp < nsp; ++sp) {
    const float *ps = p.partials + int64_t(s0 + sp) * p.slot_floats + kHeads * kDv;
    const float f = exp2f(__ldcg(ps + row) - Mu);
    lam += __ldcg(ps + kHeads + row) * f;
    lamf += __ldcg(ps + 2 * kHeads + row) * f;
  }
  const float inv = 1.f / lam;
  const int64_t orow = int64_t(b) * kHeads + row;
  for (int c = 0; c < 256; c += 32) {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
      const float *ps = p.partials + int64_t(s0 + sp) * p.slot_floats;
      const float f = exp2f(__ldcg(ps + kHeads * kDv + row) - Mu);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] += __ldcg(ps + (col0 + c + i) * kHeads + row) * f;
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) pk[i / 2] = ptx::pack_bf16(acc[i] * inv, acc[i + 1] * inv);
    uint4 *o4 = reinterpret_cast<uint4 *>(p.out + orow * kDv + col0 + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
  if (col0 == 0) p.lse[orow] = (Mx + log2f(lamf)) * kLn2;
}

int launch_mla_combine(const DecodeArgs &a) {
  if (a.shape.batch == 0) return SKD_OK;
  Params p = {};
  p.plan = a.plan;
  uint8_t *ws = static_cast<uint8_t *>(a.ws);
  p.partials = reinterpret_cast<float *>(ws + a.wl.partials);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.batch = a.shape.batch;
  p.slot_floats = a.wl.slot_floats;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.shape.batch);
  cfg.blockDim = dim3(256);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mla_combine_kernel, p, a.n_ctas) != cudaSuccess) return SKD_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace skd
