// C-ABI entry points of libskdecode (declared in include/skdecode.h):
// argument validation, workspace layout, tensor-map encoding and launches.
// Nothing here allocates device memory; every buffer belongs to the caller.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "plan_layout.h"
#include "skdecode.h"

namespace skd {
int build_plan_host(const int32_t *seqlens, int batch, int ngrp, int page_size, int n, int mode, int seg_cost,
                    int align, void *plan_out, size_t plan_bytes);

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

void *g_trace = nullptr;
bool g_pdl = true;
size_t g_trace_bytes = 0;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
}  // namespace

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, cuuint32_t rank, void *gaddr,
                      const cuuint64_t *gdim, const cuuint64_t *gstride, const cuuint32_t *box,
                      const cuuint32_t *estride, CUtensorMapSwizzle swz) {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  return g_encode(map, dt, rank, gaddr, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool pdl_enabled() { return g_pdl; }

void *trace_buffer(int n_ctas) {
  return (g_trace && g_trace_bytes >= size_t(n_ctas) * SKD_TRACE_RECORD_BYTES) ? g_trace : nullptr;
}

// rows per (request, kv head) item: every query row that reads that kv head
static int item_rows(const skd_shape_t &s) {
  return (s.num_q_heads / s.num_kv_heads) * s.q_tokens;
}

WsLayout ws_layout(const skd_shape_t &s, int n_ctas) {
  WsLayout w;
  const int hg = head_group(s.num_kv_heads);
  const int64_t items = int64_t(s.batch) * (s.num_kv_heads / hg);
  w.rows = item_rows(s);
  w.slots = 2 * int64_t(n_ctas);
  w.counters = 256;
  w.group_counters = align_up(w.counters + 4 * items, 256);
  w.partials = align_up(w.group_counters + 4 * w.slots, 256);
  w.head_floats = align_up(int64_t(w.rows) * (s.head_dim_v + 3), 4);
  w.slot_floats = w.head_floats * hg;
  w.bytes = w.partials + w.slots * w.slot_floats * 4;
  return w;
}

static int validate_shape(const skd_shape_t *s) {
  if (!s) return SKD_EINVAL;
  if (s->batch < 0 || s->q_tokens < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 ||
      s->num_q_heads % s->num_kv_heads != 0 || s->head_dim_qk < 1 || s->head_dim_v < 1 ||
      s->page_size < 1 || s->max_pages_per_req < 1 || s->num_pages < 1 ||
      s->v_row_stride < s->head_dim_v || !isfinite(s->scale))
    return SKD_EINVAL;
  if (s->page_size % kGranule != 0) return SKD_EUNSUPPORTED;
  if ((int64_t(s->v_row_stride) * 2) % 16 != 0 || (int64_t(s->head_dim_qk) * 2) % 16 != 0)
    return SKD_EINVAL;
  if (s->kind == SKD_KIND_GQA) {
    if (s->head_dim_qk != s->head_dim_v || (s->head_dim_qk != 64 && s->head_dim_qk != 128))
      return SKD_EUNSUPPORTED;
    if (item_rows(*s) > 16) return SKD_EUNSUPPORTED;
  } else if (s->kind == SKD_KIND_MLA) {
    if (s->head_dim_qk != 576 || s->head_dim_v != 512 || s->num_kv_heads != 1 ||
        s->num_q_heads != 128 || s->q_tokens != 1 || s->v_row_stride != 576)
      return SKD_EUNSUPPORTED;
  } else {
    return SKD_EINVAL;
  }
  return SKD_OK;
}

}  // namespace skd

using namespace skd;

extern "C" {

int skd_abi_version(void) { return SKD_ABI_VERSION; }

const char *skd_status_string(int st) {
  switch (st) {
    case SKD_OK: return "ok";
    case SKD_EINVAL: return "invalid argument";
    case SKD_EUNSUPPORTED: return "unsupported configuration";
    case SKD_ECUDA: return "CUDA error";
    case SKD_EPLAN: return "plan buffer too small or inconsistent";
    case SKD_ESIZE: return "workspace too small";
    default: return "unknown status";
  }
}

int skd_device_sm_count(int device, int *sm_count_out) {
  if (!sm_count_out) return SKD_EINVAL;
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return SKD_ECUDA;
  *sm_count_out = v;
  return SKD_OK;
}

int skd_default_workers(const skd_shape_t *shape, int device, int *n_out) {
  if (!shape || !n_out) return SKD_EINVAL;
  const int st = validate_shape(shape);
  if (st != SKD_OK) return st;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return SKD_ECUDA;
  if (shape->kind == SKD_KIND_GQA) {
    *n_out = sms;
    return SKD_OK;
  }
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return SKD_ECUDA;
  int n = 0;
  const int r = mla_resident_workers(&n);
  if (cudaSetDevice(cur) != cudaSuccess || r != SKD_OK) return SKD_ECUDA;
  *n_out = std::max(1, std::min(n, sms / 2));
  return SKD_OK;
}

size_t skd_plan_bytes(int batch, int num_kv_heads, int n_ctas) {
  if (batch < 0 || num_kv_heads < 1 || n_ctas < 1) return 0;
  const int ngrp = num_kv_heads / head_group(num_kv_heads);
  return size_t(plan_offsets(batch, ngrp, n_ctas).words) * 4;
}

int skd_decode_plan(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                    int n_ctas, int mode, void *plan_host, size_t plan_bytes) {
  if (num_kv_heads < 1) return SKD_EINVAL;
  return build_plan_host(seqlens_host, batch, num_kv_heads / head_group(num_kv_heads), page_size,
                         n_ctas, mode, 0, 1, plan_host, plan_bytes);
}

int skd_decode_plan_aligned(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                            int n_ctas, int seg_cost, int align, void *plan_host, size_t plan_bytes) {
  if (num_kv_heads < 1) return SKD_EINVAL;
  return build_plan_host(seqlens_host, batch, num_kv_heads / head_group(num_kv_heads), page_size,
                         n_ctas, SKD_PLAN_STREAMK, seg_cost, align, plan_host, plan_bytes);
}

int skd_decode_plan_weighted(const int32_t *seqlens_host, int batch, int num_kv_heads, int page_size,
                             int n_ctas, int seg_cost, void *plan_host, size_t plan_bytes) {
  return skd_decode_plan_aligned(seqlens_host, batch, num_kv_heads, page_size, n_ctas, seg_cost, 1, plan_host,
                                 plan_bytes);
}

int skd_decode_plan_aligned_device(const int32_t *seqlens_dev, int batch, int num_kv_heads, int page_size,
                                   int n_ctas, int seg_cost, int align, void *plan_dev, size_t plan_bytes,
                                   void *stream) {
  if ((!seqlens_dev && batch > 0) || !plan_dev || batch < 0 || num_kv_heads < 1 || n_ctas < 1)
    return SKD_EINVAL;
  if (page_size <= 0 || page_size % kGranule != 0) return SKD_EINVAL;
  if (seg_cost < 0 || seg_cost > kMaxSegCost || align < 1 || align > kMaxAlign) return SKD_EINVAL;
  if (!aligned(plan_dev, 16)) return SKD_EINVAL;
  if (plan_bytes < skd_plan_bytes(batch, num_kv_heads, n_ctas)) return SKD_EPLAN;
  return launch_plan_device(seqlens_dev, batch, num_kv_heads / head_group(num_kv_heads), n_ctas, seg_cost, align,
                            static_cast<int32_t *>(plan_dev), static_cast<cudaStream_t>(stream));
}

int skd_decode_plan_weighted_device(const int32_t *seqlens_dev, int batch, int num_kv_heads, int page_size,
                                    int n_ctas, int seg_cost, void *plan_dev, size_t plan_bytes,
                                    void *stream) {
  return skd_decode_plan_aligned_device(seqlens_dev, batch, num_kv_heads, page_size, n_ctas, seg_cost, 1,
                                        plan_dev, plan_bytes, stream);
}

int skd_decode_plan_device(const int32_t *seqlens_dev, int batch, int num_kv_heads, int page_size,
                           int n_ctas, void *plan_dev, size_t plan_bytes, void *stream) {
  return skd_decode_plan_weighted_device(seqlens_dev, batch, num_kv_heads, page_size, n_ctas, 0, plan_dev,
                                         plan_bytes, stream);
}

size_t skd_workspace_bytes(const skd_shape_t *shape, int n_ctas) {
  if (validate_shape(shape) != SKD_OK || n_ctas < 1) return 0;
  return size_t(ws_layout(*shape, n_ctas).bytes);
}

int skd_workspace_reset(void *ws, size_t ws_bytes, void *stream) {
  if (!ws || ws_bytes < 256) return SKD_EINVAL;
  // error word and counters live in front of the partial slots; clearing the
  // whole buffer keeps this independent of the shape
  if (cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SKD_ECUDA;
  return SKD_OK;
}

static int decode_common(const skd_shape_t *shape, const void *q, const void *k_pages, const void *v_pages,
                         const int32_t *page_table, const int32_t *seqlens, const void *plan_dev, int n_ctas,
                         void *ws, size_t ws_bytes, void *out, float *lse, void *stream, bool two_kernel) {
  const int st = validate_shape(shape);
  if (st != SKD_OK) return st;
  if (n_ctas < 1) return SKD_EINVAL;
  if (shape->batch == 0) return SKD_OK;
  if (!q || !k_pages || !v_pages || !page_table || !seqlens || !plan_dev || !ws || !out || !lse)
    return SKD_EINVAL;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
      !aligned(plan_dev, 16) || !aligned(ws, 256) || !aligned(page_table, 4) ||
      !aligned(seqlens, 4) || !aligned(lse, 4))
    return SKD_EINVAL;
  DecodeArgs a;
  a.shape = *shape;
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.page_table = page_table;
  a.seqlens = seqlens;
  a.plan = static_cast<const int32_t *>(plan_dev);
  a.n_ctas = n_ctas;
  a.ws = ws;
  a.wl = ws_layout(*shape, n_ctas);
  if (ws_bytes < size_t(a.wl.bytes)) return SKD_ESIZE;
  a.out = out;
  a.lse = lse;
  a.stream = static_cast<cudaStream_t>(stream);
  a.defer_merge = two_kernel;
  const bool gqa = shape->kind == SKD_KIND_GQA;
  int st2 = gqa ? launch_gqa(a) : launch_mla(a);
  if (st2 == SKD_OK && two_kernel) st2 = gqa ? launch_gqa_combine(a) : launch_mla_combine(a);
  return st2;
}

int skd_decode_attention(const skd_shape_t *shape, const void *q, const void *k_pages,
                         const void *v_pages, const int32_t *page_table, const int32_t *seqlens,
                         const void *plan_dev, int n_ctas, void *ws, size_t ws_bytes, void *out,
                         float *lse, void *stream) {
  return decode_common(shape, q, k_pages, v_pages, page_table, seqlens, plan_dev, n_ctas, ws, ws_bytes, out,
                       lse, stream, false);
}

int skd_decode_attention_split_combine(const skd_shape_t *shape, const void *q, const void *k_pages,
                                       const void *v_pages, const int32_t *page_table, const int32_t *seqlens,
                                       const void *plan_dev, int n_ctas, void *ws, size_t ws_bytes, void *out,
                                       float *lse, void *stream) {
  return decode_common(shape, q, k_pages, v_pages, page_table, seqlens, plan_dev, n_ctas, ws, ws_bytes, out,
                       lse, stream, true);
}

int skd_decode_attention_sparse(const skd_shape_t *shape, const void *q, const void *kv_pages,
                                const int32_t *page_table, const int32_t *seqlens, const int32_t *topk_idx,
                                int topk_stride, const int32_t *topk_len, const void *plan_dev, int n_ctas,
                                void *ws, size_t ws_bytes, void *out, float *lse, void *stream) {
  const int st = validate_shape(shape);
  if (st != SKD_OK) return st;
  if (shape->kind != SKD_KIND_MLA) return SKD_EUNSUPPORTED;
  if (n_ctas < 1 || topk_stride < 1) return SKD_EINVAL;
  if (shape->batch == 0) return SKD_OK;
  if (!q || !kv_pages || !page_table || !seqlens || !topk_idx || !topk_len || !plan_dev || !ws || !out || !lse)
    return SKD_EINVAL;
  if (!aligned(q, 16) || !aligned(kv_pages, 16) || !aligned(out, 16) || !aligned(plan_dev, 16) ||
      !aligned(ws, 256) || !aligned(page_table, 4) || !aligned(seqlens, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_len, 4) || !aligned(lse, 4))
    return SKD_EINVAL;
  DecodeArgs a;
  a.shape = *shape;
  a.q = q;
  a.k = kv_pages;
  a.v = kv_pages;
  a.page_table = page_table;
  a.seqlens = seqlens;
  a.plan = static_cast<const int32_t *>(plan_dev);
  a.n_ctas = n_ctas;
  a.ws = ws;
  a.wl = ws_layout(*shape, n_ctas);
  if (ws_bytes < size_t(a.wl.bytes)) return SKD_ESIZE;
  a.out = out;
  a.lse = lse;
  a.stream = static_cast<cudaStream_t>(stream);
  a.topk = topk_idx;
  a.topk_len = topk_len;
  a.topk_stride = topk_stride;
  return launch_mla(a);
}

int skd_gather_rows(void *dst, const void *src, const int32_t *src_rows, int64_t n_rows, int64_t row_bytes,
                    void *stream) {
  if (n_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return SKD_EINVAL;
  if (n_rows == 0) return SKD_OK;
  if (!dst || !src || !src_rows || !aligned(dst, 16) || !aligned(src, 16) || !aligned(src_rows, 4))
    return SKD_EINVAL;
  return launch_gather_rows(dst, src, src_rows, n_rows, row_bytes, static_cast<cudaStream_t>(stream));
}

int skd_merge_states(const void *out_a, const float *lse_a, const int32_t *a_rows, const void *out_b,
                     const float *lse_b, const int32_t *b_rows, void *out, float *lse, int64_t n_rows,
                     int head_dim_v, void *stream) {
  if (n_rows < 0 || head_dim_v <= 0 || head_dim_v % 8 != 0) return SKD_EINVAL;
  if (n_rows == 0) return SKD_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse || !aligned(out_a, 16) || !aligned(out_b, 16) ||
      !aligned(out, 16) || !aligned(lse_a, 4) || !aligned(lse_b, 4) || !aligned(lse, 4) ||
      (a_rows && !aligned(a_rows, 4)) || (b_rows && !aligned(b_rows, 4)))
    return SKD_EINVAL;
  return launch_merge_states(out_a, lse_a, a_rows, out_b, lse_b, b_rows, out, lse, n_rows, head_dim_v,
                             static_cast<cudaStream_t>(stream));
}

int skd_set_pdl(int enable) {
  g_pdl = enable != 0;
  return SKD_OK;
}

int skd_trace_enable(void *trace_dev, size_t bytes) {
  if (trace_dev && !aligned(trace_dev, 8)) return SKD_EINVAL;
  g_trace = trace_dev;
  g_trace_bytes = trace_dev ? bytes : 0;
  return SKD_OK;
}

int skd_read_error(const void *ws, int32_t *err_out, void *stream) {
  if (!ws || !err_out) return SKD_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(err_out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SKD_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SKD_ECUDA;
  return SKD_OK;
}

}  // extern "C"
