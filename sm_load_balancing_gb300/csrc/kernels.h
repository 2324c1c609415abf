// Internal launcher interface between the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "skdecode.h"

namespace skd {

// Workspace layout: [0,256) error word; item counters (one int32 per
// (request, kv-head group) item); merge-tree counters (one int32 per slot);
// partial-state slots (2 per CTA). A slot holds, for each head of the group, a
// block of head_floats floats: O[rows][Dv], m[rows], l[rows], lf[rows] (m in
// log2 units of the scaled score; l sums the bf16-rounded probabilities that
// entered P.V, lf the fp32 ones).
struct WsLayout {
  int64_t counters, group_counters, partials, slot_floats, head_floats, slots, bytes;
  int rows;
};
WsLayout ws_layout(const skd_shape_t &s, int n_ctas);

struct DecodeArgs {
  skd_shape_t shape;
  const void *q, *k, *v;
  const int32_t *page_table, *seqlens, *plan;
  int n_ctas;
  void *ws;
  WsLayout wl;
  void *out;
  float *lse;
  cudaStream_t stream;
  bool defer_merge = false;  // splits only write their partial states (two-kernel comparator)
  // sparse MLA: listed cache positions [batch][topk_stride] and list lengths (null: dense)
  const int32_t *topk = nullptr, *topk_len = nullptr;
  int topk_stride = 0;
};

int launch_gqa(const DecodeArgs &a);
int launch_mla(const DecodeArgs &a);
// MLA workers (2-CTA clusters) that can be resident at once on the current device
int mla_resident_workers(int *n);
// the comparator's second kernel: merge every split item's partial states
int launch_gqa_combine(const DecodeArgs &a);
int launch_mla_combine(const DecodeArgs &a);
// compose.cu: dst row i = src row src_rows[i] (zeros for a negative index)
int launch_gather_rows(void *dst, const void *src, const int32_t *src_rows, int64_t n_rows, int64_t row_bytes,
                       cudaStream_t stream);
// compose.cu: merge two attention results (out bf16, lse) over disjoint key sets, row by row
int launch_merge_states(const void *out_a, const float *lse_a, const int32_t *a_rows, const void *out_b,
                        const float *lse_b, const int32_t *b_rows, void *out, float *lse, int64_t n_rows,
                        int head_dim_v, cudaStream_t stream);
int launch_plan_device(const int32_t *seqlens, int batch, int ngrp, int n_ctas, int seg_cost, int align, int32_t *plan,
                       cudaStream_t stream);

// cuTensorMapEncodeTiled, looked up through the runtime (no libcuda link).
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, cuuint32_t rank, void *gaddr,
                      const cuuint64_t *gdim, const cuuint64_t *gstride, const cuuint32_t *box,
                      const cuuint32_t *estride, CUtensorMapSwizzle swz);

// Launch the attention kernels with programmatic dependent launch (the kernel
// may start while the previous kernel of the stream finishes; it waits with
// griddepcontrol.wait before reading any input). Set by skd_set_pdl.
bool pdl_enabled();

// Per-CTA timing records enabled by skd_trace_enable (nullptr when off or when
// the buffer is too small for n_ctas records).
void *trace_buffer(int n_ctas);

// Bounded device waits give up after this many SM cycles (about one second).
constexpr long long kWaitCycles = 2000000000LL;

}  // namespace skd
