// Kernels that compose decode launches: gather query rows into a batch of
// virtual requests, and merge two attention results over disjoint key sets.
//
// Shared-prefix decode ("MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）",
// results, shared-prefix decode (Fig. 11); its core method reduces partial
// states of one query row computed over different key ranges) reads a prefix
// that several requests share once for all of them and combines that state
// with each request's own suffix state. Softmax attention over a union of
// disjoint key sets A and B follows from the two results alone: with
// M = max(lse_A, lse_B) and w_X = exp(lse_X - M),
//   out = (w_A out_A + w_B out_B) / (w_A + w_B),  lse = M + ln(w_A + w_B).
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"

namespace skd {
namespace {

// dst row i = src row src_rows[i], or zeros when src_rows[i] < 0; rows of
// row_bytes (a multiple of 16), one warp per row
__global__ void gather_rows_kernel(uint4 *dst, const uint4 *src, const int32_t *src_rows, int64_t n_rows,
                                   int64_t row_vec) {
  const int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n_rows) return;
  const int32_t r = src_rows[i];
  uint4 *d = dst + i * row_vec;
  if (r < 0) {
    for (int64_t c = lane; c < row_vec; c += 32) d[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4 *s = src + int64_t(r) * row_vec;
  for (int64_t c = lane; c < row_vec; c += 32) d[c] = __ldg(s + c);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&t);
}

// row r: state A = (out_a, lse_a) row a_rows[r], state B = (out_b, lse_b)
// row b_rows[r] (a negative entry: no such state; a null map: row r); result
// into row r of out / lse (which may be B's arrays when b_rows is null). One
// warp per row, 8 values per lane and step.
__global__ void merge_states_kernel(const uint4 *out_a, const float *lse_a, const int32_t *a_rows, const uint4 *out_b,
                                    const float *lse_b, const int32_t *b_rows, uint4 *out, float *lse, int64_t n_rows,
                                    int vec) {
  const int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  const int64_t ra = a_rows ? int64_t(a_rows[r]) : r, rb = b_rows ? int64_t(b_rows[r]) : r;
  const float la = ra >= 0 ? lse_a[ra] : -INFINITY, lb = rb >= 0 ? lse_b[rb] : -INFINITY;
  const float M = fmaxf(la, lb);
  float wa = 0.f, wb = 0.f, inv = 0.f;
  if (M != -INFINITY) {
    wa = la == -INFINITY ? 0.f : expf(la - M);
    wb = lb == -INFINITY ? 0.f : expf(lb - M);
    inv = 1.f / (wa + wb);
  }
  for (int c = lane; c < vec; c += 32) {
    const uint4 b = wb != 0.f ? out_b[rb * vec + c] : make_uint4(0, 0, 0, 0);
    const uint4 a = wa != 0.f ? out_a[ra * vec + c] : make_uint4(0, 0, 0, 0);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = pack_bf16((wa * bf16_lo(av[k]) + wb * bf16_lo(bv[k])) * inv,
                       (wa * bf16_hi(av[k]) + wb * bf16_hi(bv[k])) * inv);
    out[r * vec + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncwarp();  // every lane has read lse_b[r] (lse may be the same array)
  if (lane == 0) lse[r] = M == -INFINITY ? -INFINITY : M + logf(wa + wb);
}

}  // namespace

int launch_gather_rows(void *dst, const void *src, const int32_t *src_rows, int64_t n_rows, int64_t row_bytes,
                       cudaStream_t stream) {
  if (n_rows == 0) return SKD_OK;
  const int64_t threads = n_rows * 32;
  gather_rows_kernel<<<unsigned((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), src_rows, n_rows, row_bytes / 16);
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

int launch_merge_states(const void *out_a, const float *lse_a, const int32_t *a_rows, const void *out_b,
                        const float *lse_b, const int32_t *b_rows, void *out, float *lse, int64_t n_rows,
                        int head_dim_v, cudaStream_t stream) {
  if (n_rows == 0) return SKD_OK;
  const int64_t threads = n_rows * 32;
  merge_states_kernel<<<unsigned((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const uint4 *>(out_a), lse_a, a_rows, static_cast<const uint4 *>(out_b), lse_b, b_rows,
      static_cast<uint4 *>(out), lse, n_rows, head_dim_v / 8);
  return cudaGetLastError() == cudaSuccess ? SKD_OK : SKD_ECUDA;
}

}  // namespace skd
