/*
 * skdecode -- Stream-K split-KV decode attention over a paged KV cache, for
 * sm_103a (GB300). C ABI: plain pointers and sizes, no framework types.
 *
 * What the library computes (the passages it follows):
 *   - attention itself: exact softmax attention, QK^T -> mask -> softmax -> xV,
 *     streamed with an online softmax so no score matrix is written to HBM
 *     ("GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 6.3 and Q8);
 *   - the work split: the batch's KV tokens are cut into as many near-equal
 *     chunks as there are CTAs and launched as one wave (triton.csdn.net Q&A
 *     on waves and FlashMLA's Stream-K, closing summary);
 *   - the reduction: partial softmax states of the splits of one (request,
 *     kv head) are merged inside the same kernel as soon as the last split is
 *     done -- no separate combine kernel and no wait for the slowest SM
 *     ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", key observations and
 *     core method: just-in-time reduction);
 *   - the split is chosen at run time from the real sequence lengths
 *     (same page, core method).
 *
 * Conventions for every call
 *   - The caller owns and allocates every buffer; the library allocates no
 *     device memory. "device" pointers are CUDA global-memory addresses on the
 *     current device; "host" pointers are ordinary CPU memory.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream. Calls that take a stream only enqueue work on it.
 *   - Every call returns an skd_status (SKD_OK == 0) and never throws.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (2 bytes, little endian).
 *
 * Tensor layouts (row-major, all contiguous unless a stride is given)
 *   q          bf16   [B][T][Hq][Dk]
 *   k_pages    bf16   [NP][P][Hkv][Dk]           (token-major pages, "NHD")
 *   v_pages    bf16   rows of Dv values; row (page, slot, kv head) starts at
 *                     element ((page*P + slot)*Hkv + head) * v_row_stride.
 *                     GQA: its own buffer [NP][P][Hkv][Dv], v_row_stride = Dv.
 *                     MLA (absorbed): v_pages == k_pages, Hkv = 1,
 *                     v_row_stride = Dk = 576, Dv = 512 (V = the first 512
 *                     columns of the shared latent row).
 *   page_table int32  [B][max_pages_per_req]; entry j of request b is the
 *                     physical page holding tokens [j*P, (j+1)*P).
 *   seqlens    int32  [B]; KV tokens of request b, the T new ones included.
 *   out        bf16   [B][T][Hq][Dv]
 *   lse        fp32   [B][T][Hq]; natural log of sum_j exp(scale * q.k_j).
 *
 * Semantics where the pages are silent
 *   - query head h reads kv head h / (Hq/Hkv);
 *   - the T query tokens are the last T cache positions; with `causal` query
 *     token t sees keys j <= L - T + t;
 *   - L == 0 gives out = 0 and lse = -inf;
 *   - causal with 0 < L < T is an input error.
 */
#ifndef SKDECODE_H_
#define SKDECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKD_ABI_VERSION 1
/* KV tokens per planning granule; split points fall on multiples of it. */
#define SKD_GRANULE 16

typedef enum skd_status {
  SKD_OK = 0,
  SKD_EINVAL = 1,        /* bad argument: null pointer, negative size, misaligned pointer */
  SKD_EUNSUPPORTED = 2,  /* valid but not implemented (head dims, page size, group size) */
  SKD_ECUDA = 3,         /* a CUDA runtime or driver call failed */
  SKD_EPLAN = 4,         /* plan buffer too small or inconsistent with the call */
  SKD_ESIZE = 5          /* workspace too small */
} skd_status;

typedef enum skd_kind { SKD_KIND_GQA = 0, SKD_KIND_MLA = 1 } skd_kind;

typedef enum skd_plan_mode {
  SKD_PLAN_STREAMK = 0,      /* one-wave near-equal split (the method) */
  SKD_PLAN_ROUND_ROBIN = 1,  /* whole (request, kv head) items dealt in turn; comparator */
  SKD_PLAN_FIXED_SPLIT = 2   /* every item cut into the same number of splits, merged by a
                                separate combine kernel (skd_decode_attention_split_combine);
                                the two-kernel split-KV comparator */
} skd_plan_mode;

/* Bits of the device error word (see skd_read_error). */
#define SKD_DEVERR_PLAN 0x1      /* plan header does not match the launch */
#define SKD_DEVERR_SEQLEN 0x2    /* a seqlen disagrees with the plan or the page table size */
#define SKD_DEVERR_PAGE 0x4      /* a page id outside [0, num_pages) */
#define SKD_DEVERR_TIMEOUT 0x8   /* a bounded wait inside the kernel gave up */
#define SKD_DEVERR_INDEX 0x10    /* sparse: a listed position outside [0, seqlens[b]) */

typedef struct skd_shape {
  int32_t batch;             /* B >= 0 */
  int32_t q_tokens;          /* T >= 1 */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv, divides Hq */
  int32_t head_dim_qk;       /* Dk: GQA 64 or 128; MLA 576 */
  int32_t head_dim_v;        /* Dv: GQA == Dk; MLA 512 */
  int32_t page_size;         /* P, a multiple of SKD_GRANULE */
  int32_t max_pages_per_req; /* columns of page_table */
  int32_t num_pages;         /* NP, pages in k_pages (and v_pages) */
  int32_t v_row_stride;      /* elements between consecutive V rows (>= Dv) */
  float scale;               /* softmax scale applied to q.k (required) */
  int32_t causal;            /* 1: mask among the T new tokens */
  int32_t kind;              /* skd_kind */
} skd_shape_t;

/* ABI version of the loaded library (SKD_ABI_VERSION). */
int skd_abi_version(void);

/* Static text for a status code. */
const char *skd_status_string(int status);

/* Number of SMs of CUDA device `device` (one persistent CTA per SM is the
 * intended grid). */
int skd_device_sm_count(int device, int *sm_count_out);

/* Workers (n_ctas) for one wave of the decode kernel of `shape` on CUDA device
 * `device`: GQA: one CTA per SM; absorbed MLA: a worker is a cluster of 2 CTAs
 * (a score SM and a value SM), so the number of such clusters that fit on the
 * device at once (at most SMs / 2). Any n_ctas >= 1 is valid for the
 * decode calls; fewer than this leaves SMs idle, more runs in several waves.
 * Errors: SKD_EINVAL (null pointer or invalid shape), SKD_ECUDA. */
int skd_default_workers(const skd_shape_t *shape, int device, int *n_out);

/* ---- planner ----------------------------------------------------------- */

/* Bytes of a plan for `batch` requests, `num_kv_heads` heads, `n_ctas` CTAs.
 * Returns 0 for invalid arguments. The plan has a fixed size for fixed
 * (batch, num_kv_heads, n_ctas), so it can live in a graph-captured buffer. */
size_t skd_plan_bytes(int batch, int num_kv_heads, int n_ctas);

/* Host planner (pure function, no CUDA call). Splits the KV-token work of the
 * batch into `n_ctas` chunks (mode SKD_PLAN_STREAMK) and writes the per-CTA
 * segment list to `plan_host` (plan_bytes >= skd_plan_bytes(...)); copy it to
 * the device before skd_decode_attention.
 * The kv heads of a request are processed in groups of HG heads, HG = the
 * largest divisor of num_kv_heads not above 8 (so NGRP = num_kv_heads / HG
 * groups; MLA: 1). Work item i = b*NGRP + g has ceil(seqlens[b] / SKD_GRANULE)
 * granules (a granule = SKD_GRANULE tokens of all HG heads); chunk c is
 * granules [floor(c*G/n), floor((c+1)*G/n)) of all items in order, cut at item
 * boundaries. seqlens_host: host int32[batch]; page_size must be a multiple
 * of SKD_GRANULE. Errors: SKD_EINVAL (null pointer, n_ctas <= 0, negative
 * seqlen, page_size), SKD_EPLAN (buffer too small, more than 2^31-1 granules). */
int skd_decode_plan(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                    int n_ctas, int mode, void *plan_host, size_t plan_bytes);

/* Device planner: the same plan, byte for byte, computed on the GPU from device
 * seqlens by one kernel enqueued on `stream` (no host synchronisation, so it
 * can be captured in a CUDA graph together with skd_decode_attention).
 * seqlens_dev: device int32[batch]; plan_dev: device buffer of plan_bytes.
 * Only mode SKD_PLAN_STREAMK. Bad seqlens (negative) set SKD_DEVERR_SEQLEN in
 * the plan header's error field, which skd_decode_attention propagates. */
int skd_decode_plan_device(const int32_t *seqlens_dev, int batch, int num_kv_heads,
                           int page_size, int n_ctas, void *plan_dev, size_t plan_bytes,
                           void *stream);

/* Weighted Stream-K split (an extension: the pages charge nothing per
 * segment). Every non-empty work item is preceded by `seg_cost` virtual
 * granules that carry no tokens, standing for the fixed time a CTA spends per
 * segment (loading the item's queries, writing its output or partial state);
 * the equal split of triton.csdn.net's closing summary then runs over the
 * virtual total, so a CTA whose range crosses many item boundaries gets fewer
 * tokens. seg_cost = 0 gives exactly skd_decode_plan's STREAMK plan. Host and
 * device variants produce identical bytes. 0 <= seg_cost <= 65536, else
 * SKD_EINVAL; other arguments and errors as skd_decode_plan /
 * skd_decode_plan_device. The value used is stored in the plan header. */
int skd_decode_plan_weighted(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                             int n_ctas, int seg_cost, void *plan_host, size_t plan_bytes);
int skd_decode_plan_weighted_device(const int32_t *seqlens_dev, int batch, int num_kv_heads, int page_size,
                                    int n_ctas, int seg_cost, void *plan_dev, size_t plan_bytes,
                                    void *stream);

/* Weighted split with aligned split points (a second extension). The equal
 * split runs over cut units of `align` granules instead of single granules:
 * work item i has ceil(seqlens[b] / (SKD_GRANULE * align)) units, preceded
 * (when non-empty) by ceil(seg_cost / align) virtual units, and every split
 * point inside an item falls on a multiple of SKD_GRANULE * align tokens. A
 * kernel that reads an item in whole blocks of that many tokens (the MLA
 * kernel: 64 tokens, align = 4) then never reads one block in two splits.
 * align = 1 gives exactly skd_decode_plan_weighted's plan. 1 <= align <= 64,
 * else SKD_EINVAL; other arguments and errors as skd_decode_plan_weighted /
 * skd_decode_plan_weighted_device. Host and device variants produce identical
 * bytes; align is stored in the plan header. */
int skd_decode_plan_aligned(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                            int n_ctas, int seg_cost, int align, void *plan_host, size_t plan_bytes);
int skd_decode_plan_aligned_device(const int32_t *seqlens_dev, int batch, int num_kv_heads, int page_size,
                                   int n_ctas, int seg_cost, int align, void *plan_dev, size_t plan_bytes,
                                   void *stream);

/* The two-kernel split-KV comparator (the design the pages measure MeldKernel
 * against: split-KV with fixed splits and a separate combine pass). Same
 * arguments as skd_decode_attention; plan_dev should come from skd_decode_plan
 * with mode SKD_PLAN_FIXED_SPLIT. The attention kernel writes every split's
 * partial state (m, l, acc) to the workspace without counting arrivals, then a
 * second kernel (one CTA per request and kv-head group) merges each item's
 * splits in split order and writes out / lse. Two launches on `stream`. */
int skd_decode_attention_split_combine(const skd_shape_t *shape, const void *q, const void *k_pages,
                                       const void *v_pages, const int32_t *page_table, const int32_t *seqlens,
                                       const void *plan_dev, int n_ctas, void *ws, size_t ws_bytes, void *out,
                                       float *lse, void *stream);

/* Sparse (top-k) absorbed-MLA decode attention: request b attends only to
 * the cache positions topk_idx[b * topk_stride + i], i < topk_len[b] (device
 * int32 arrays; positions in [0, seqlens[b]), any order, a repeated position
 * counts as two keys, no causal mask; topk_len[b] == 0 gives out = 0 and
 * lse = -inf). This is the sparse MLA step that follows an indexer's top-k in
 * the GLM-5.2-FP8 decode article (tahou.com: summary; related-work paragraph
 * on TileRT gathering the sparse KV rows by the top-2048 indices), run through
 * the same Stream-K split and just-in-time merge: build the plan with the
 * planner over topk_len (as the per-request lengths), kv heads = 1. The kernel
 * gathers each listed latent row (576 bf16, row stride shape->v_row_stride)
 * with 16-byte copies. shape->kind must be SKD_KIND_MLA (else SKD_EUNSUPPORTED);
 * other arguments, ownership and errors as skd_decode_attention; a listed
 * position outside [0, seqlens[b]) sets SKD_DEVERR_INDEX (that key is then
 * position 0), topk_len[b] > topk_stride sets SKD_DEVERR_SEQLEN. */
int skd_decode_attention_sparse(const skd_shape_t *shape, const void *q, const void *kv_pages,
                                const int32_t *page_table, const int32_t *seqlens, const int32_t *topk_idx,
                                int topk_stride, const int32_t *topk_len, const void *plan_dev, int n_ctas,
                                void *ws, size_t ws_bytes, void *out, float *lse, void *stream);

/* ---- composing decode launches (shared-prefix decode) ------------------ */

/* dst row i = src row src_rows[i] for i < n_rows, a row of zeros where
 * src_rows[i] < 0. Rows are row_bytes long (a multiple of 16); dst and src
 * 16-byte aligned, src_rows int32 on the device. Used to stack the query rows
 * of requests that share a prefix into one virtual request. Asynchronous on
 * `stream`; errors: SKD_EINVAL (sizes, null or misaligned pointers), SKD_ECUDA. */
int skd_gather_rows(void *dst, const void *src, const int32_t *src_rows, int64_t n_rows, int64_t row_bytes,
                    void *stream);

/* Merge two attention results of the same query rows over disjoint key sets
 * A and B (the reduction of partial states in "MeldKernel：动态负载下跨 SM 融合内核
 * （SOSP 2026）", core method; used for its shared-prefix decode, Fig. 11):
 * with M = max(lse_A, lse_B), w_X = exp(lse_X - M):
 *   out = (w_A out_A + w_B out_B) / (w_A + w_B),  lse = M + ln(w_A + w_B),
 * lse in natural-log units as skd_decode_attention writes it; both empty
 * (lse = -inf) gives out = 0, lse = -inf. Row r of the result takes state A
 * from row a_rows[r] of out_a / lse_a and state B from row b_rows[r] of
 * out_b / lse_b (a negative entry: no such state; a NULL map: row r). out
 * rows are bf16 [n_rows][head_dim_v] (head_dim_v a multiple of 8), lse fp32;
 * out / lse may be out_b / lse_b when b_rows is NULL. Asynchronous; errors:
 * SKD_EINVAL, SKD_ECUDA. */
int skd_merge_states(const void *out_a, const float *lse_a, const int32_t *a_rows, const void *out_b,
                     const float *lse_b, const int32_t *b_rows, void *out, float *lse, int64_t n_rows,
                     int head_dim_v, void *stream);

/* Launch option (process-wide, default on): launch the attention kernel with
 * programmatic dependent launch, so that it can be scheduled while the
 * previous kernel of the stream (typically skd_decode_plan_device, which
 * signals its dependents as soon as it starts) is still running; the kernel
 * waits for that grid to complete before reading any input, so results do not
 * change. This is the launch-overlap idea of "GPU Kernel、异步 Launch、Stream 与
 * 融合 Kernel 全解" (section 7, launch gaps in a decode step). 0 turns it off.
 * Always SKD_OK. */
int skd_set_pdl(int enable);

/* ---- workspace --------------------------------------------------------- */

/* Bytes of the workspace skd_decode_attention needs for this shape and grid:
 * an error word, one arrival counter per work item (request, kv-head group),
 * one merge-tree counter per split slot and room for the partial softmax
 * states (m, l, acc) of up to 2*n_ctas splits. 0 if invalid. */
size_t skd_workspace_bytes(const skd_shape_t *shape, int n_ctas);

/* Zero the error word and all counters (enqueued on `stream`). Needed once
 * after allocation and after any call that set a device error; the kernel
 * itself returns every counter to zero after each successful call. */
int skd_workspace_reset(void *ws_dev, size_t ws_bytes, void *stream);

/* ---- the hot path ------------------------------------------------------ */

/* Decode attention for the whole batch in one kernel launch of `n_ctas`
 * persistent CTAs (the plan's CTA count) on `stream`. All tensor pointers are
 * device pointers in the layouts above and must be 16-byte aligned; the plan
 * (device copy) must have been built for shape->batch, shape->num_kv_heads and
 * n_ctas. Asynchronous: returns after the launch. Errors detected on the host:
 * SKD_EINVAL, SKD_EUNSUPPORTED, SKD_ESIZE, SKD_ECUDA (launch failure).
 * Errors detected on the device set bits of the workspace error word
 * (SKD_DEVERR_*); out and lse are then unspecified. Supported now:
 * kind GQA with Dk == Dv in {64, 128} and (Hq/Hkv)*T <= 16;
 * kind MLA with Dk 576, Dv 512, Hq 128, Hkv 1, T 1. */
int skd_decode_attention(const skd_shape_t *shape, const void *q, const void *k_pages,
                         const void *v_pages, const int32_t *page_table, const int32_t *seqlens,
                         const void *plan_dev, int n_ctas, void *ws_dev, size_t ws_bytes,
                         void *out, float *lse, void *stream);

/* Copy the device error word to *err_out (synchronises `stream`). */
int skd_read_error(const void *ws_dev, int32_t *err_out, void *stream);

/* Allocation-free variant of skd_decode_attention (GQA only), for callers
 * that cannot allocate device memory for a workspace: operator plugins whose
 * fixed interface has no scratch argument, or runtimes whose device memory is
 * planned up front and may not grow. The pages have no counterpart; this is an
 * interface convenience. The workspace is a fixed 32 MiB module-scope device
 * array that every GPU loading this library holds until the process exits.
 * Arguments are those of skd_decode_attention without ws/ws_bytes; the caller
 * still owns q, the cache, page table, seqlens, plan, out and lse.
 * Errors: SKD_ESIZE when skd_workspace_bytes(shape, n_ctas) exceeds 32 MiB
 * (nothing is enqueued); SKD_EUNSUPPORTED for MLA; SKD_ECUDA if the array's
 * device address cannot be obtained. The first call on a device looks that
 * address up (cudaGetSymbolAddress), so make it before any stream capture.
 * Each call clears the array's error word and counters on `stream`, then
 * launches. All calls share the one array, which keeps the last call's
 * contents: calls that overlap on the GPU (other streams, other threads)
 * race and give wrong results; serialise them. Device-side error bits land
 * in the shared array and are not reported; use skd_decode_attention with a
 * workspace to diagnose. */
int skd_decode_attention_noalloc(const skd_shape_t *shape, const void *q, const void *k_pages,
                                 const void *v_pages, const int32_t *page_table,
                                 const int32_t *seqlens, const void *plan_dev, int n_ctas, void *out,
                                 float *lse, void *stream);

/* ---- diagnostics ------------------------------------------------------- */

/* Per-CTA execution trace, after the GLM-5.2 decode article's Kineto analysis
 * of how busy the SMs are (duration-weighted SM busy fraction, idle bubbles).
 * While enabled (trace_dev != NULL) every decode-attention launch adds, for CTA
 * c, SKD_TRACE_RECORD_BYTES at trace_dev + c*SKD_TRACE_RECORD_BYTES: int64
 * words {0: %globaltimer ns at start, 1: ns at end, 2: consumer cycles spent
 * waiting for data (summed over consumer warps), 3: consumer cycles in total
 * (summed), 4: producer cycles waiting for free stages, 5: producer cycles in
 * total, 6: segments, 7: pipeline stages, 8: SM id, 9: consumer cycles spent
 * publishing and merging partial states (summed), 10: final merges, 11:
 * merge-tree node merges, 12..15: reserved}. Words 2, 3, 7, 9, 10 and 11 are
 * accumulated with atomics: zero the buffer before each launch. An absorbed-MLA
 * launch writes 2 records per worker (its cluster ranks: 0 score, 1 value):
 * {0, 1 as above, 2..11: cycles its warps spent waiting, summed per barrier
 * kind, 14: segments, 15: SM id}. A buffer smaller than n_ctas records
 * (2 n_ctas for MLA) disables tracing for that launch. Process-wide setting, not
 * thread-safe; pass NULL to disable. Errors: SKD_EINVAL (misaligned pointer). */
#define SKD_TRACE_RECORD_BYTES 128
int skd_trace_enable(void *trace_dev, size_t bytes);

#ifdef __cplusplus
}
#endif
#endif /* SKDECODE_H_ */
