/*
 * fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests, the smoke check and the CPU-baseline leg of the benchmark may
 * load this file's library. It shares no code, header or constant with the
 * CUDA path.
 *
 * What it computes is plain softmax attention written out from its definition,
 * with no splits, no blocking and no online rescaling:
 *   "GPU Kernel、异步 Launch、Stream 与融合 Kernel 全解", section 6.3 and Q8:
 *   attention is QK^T -> mask -> softmax -> xV (FlashAttention only fuses and
 *   reorders these steps; its result is the exact softmax attention).
 *   "MeldKernel：动态负载下跨 SM 融合内核（SOSP 2026）", key observations and core
 *   method: split-KV decoding followed by a reduction of the partial outputs;
 *   the merged result is the unsplit attention, which is what this file gives.
 *
 * Readings where the pages are silent (the same ones the CUDA path follows):
 *   - query head h uses kv head h / (Hq / Hkv) (contiguous grouping);
 *   - the T new tokens are the last T positions of the cache; with causal
 *     masking query token t sees keys j <= L - T + t;
 *   - lse is the natural log of the sum of exp(scale * q.k) over visible keys;
 *   - a request with L == 0 yields out = 0 and lse = -inf;
 *   - with the absorbed-MLA layout V is the first Dv columns of the K row
 *     (v_row_stride = Dk, v pointer = k pointer).
 *
 * Every bf16 input is widened exactly to double; all arithmetic is double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Returns 0 on success, or a negative code:
 *   -1  bad shape argument
 *   -2  seqlen above max_pages * page_size, or negative
 *   -3  page id outside [0, num_pages)
 *   -4  causal with 0 < seqlen < T (a query token would see no key)
 *
 * rows: optional list of flattened row ids ((b*T + t)*Hq + h); NULL = all rows.
 * out:  [n_rows][Dv] doubles; lse: [n_rows] doubles.
 */
int oracle_decode_f64(int B, int T, int Hq, int Hkv, int Dk, int Dv, int P, int max_pages,
                      int num_pages, int causal, double scale,
                      const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      long long v_row_stride, const int32_t *page_table, const int32_t *seqlens,
                      const int64_t *rows, long long n_rows, double *out, double *lse) {
    if (B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Dk <= 0 || Dv <= 0 || P <= 0 ||
        max_pages <= 0 || v_row_stride < Dv)
        return -1;
    const int G = Hq / Hkv;
    const long long total_rows = (long long)B * T * Hq;
    if (rows == NULL) n_rows = total_rows;

    /* input checks first, so that a bad case yields no partial output */
    for (int b = 0; b < B; ++b) {
        int L = seqlens[b];
        if (L < 0 || (long long)L > (long long)max_pages * P) return -2;
        if (causal && L > 0 && L < T) return -4;
        for (int j = 0; j < (L + P - 1) / P; ++j) {
            int pg = page_table[(long long)b * max_pages + j];
            if (pg < 0 || pg >= num_pages) return -3;
        }
    }

    int err = 0;
#pragma omp parallel
    {
        double *sig = NULL;
        long long cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (long long i = 0; i < n_rows; ++i) {
            long long r = rows ? rows[i] : i;
            if (r < 0 || r >= total_rows) {
#pragma omp atomic write
                err = -1;
                continue;
            }
            const int h = (int)(r % Hq);
            const int t = (int)((r / Hq) % T);
            const int b = (int)(r / ((long long)Hq * T));
            const int g = h / G;
            const int L = seqlens[b];
            /* number of visible keys for this query token */
            long long n = L;
            if (causal && L > 0) n = (long long)L - T + t + 1;
            double *o = out + i * (long long)Dv;
            for (int d = 0; d < Dv; ++d) o[d] = 0.0;
            if (n <= 0) {
                lse[i] = -INFINITY;
                continue;
            }
            if (n > cap) {
                free(sig);
                cap = n;
                sig = (double *)malloc(sizeof(double) * (size_t)cap);
            }
            const uint16_t *qr = q + r * (long long)Dk;
            /* scores sigma_j = scale * sum_d q[d] k_j[d] */
            for (long long j = 0; j < n; ++j) {
                int pg = page_table[(long long)b * max_pages + (int)(j / P)];
                int s = (int)(j % P);
                const uint16_t *kr = k_pages + (((long long)pg * P + s) * Hkv + g) * (long long)Dk;
                double acc = 0.0;
                for (int d = 0; d < Dk; ++d) acc += bf16_to_f64(qr[d]) * bf16_to_f64(kr[d]);
                sig[j] = scale * acc;
            }
            double mu = -INFINITY;
            for (long long j = 0; j < n; ++j)
                if (sig[j] > mu) mu = sig[j];
            double Z = 0.0;
            for (long long j = 0; j < n; ++j) Z += exp(sig[j] - mu);
            for (long long j = 0; j < n; ++j) {
                double w = exp(sig[j] - mu) / Z;
                int pg = page_table[(long long)b * max_pages + (int)(j / P)];
                int s = (int)(j % P);
                const uint16_t *vr = v_pages + (((long long)pg * P + s) * Hkv + g) * v_row_stride;
                for (int d = 0; d < Dv; ++d) o[d] += w * bf16_to_f64(vr[d]);
            }
            lse[i] = mu + log(Z);
        }
        free(sig);
    }
    return err;
}

/* Sparse (top-k) attention: row (b, t, h) attends to the multiset of cache
 * positions {topk_idx[b][i] : 0 <= i < topk_len[b]} and to nothing else -- the
 * plain softmax attention of the definition above restricted to the keys an
 * indexer selected. The GLM-5.2-FP8 decode article (tahou.com; summary and the
 * related-work paragraph on TileRT) has the layer continue with TopK and
 * Sparse FlashMLA, whose ranks gather the sparse KV rows named by the top-2048
 * indices; the pages give no formula, so this is the plain reading. A position
 * listed twice counts as two keys; no causal mask is applied (the selection
 * decides visibility); topk_len[b] == 0 gives out = 0 and lse = -inf. Keys are
 * summed in list order.
 *
 * Extra error codes:
 *   -5  topk_len[b] outside [0, topk_stride]
 *   -6  a listed position outside [0, seqlens[b])
 */
int oracle_decode_sparse_f64(int B, int T, int Hq, int Hkv, int Dk, int Dv, int P, int max_pages,
                             int num_pages, double scale, const uint16_t *q, const uint16_t *k_pages,
                             const uint16_t *v_pages, long long v_row_stride, const int32_t *page_table,
                             const int32_t *seqlens, const int32_t *topk_idx, int topk_stride,
                             const int32_t *topk_len, const int64_t *rows, long long n_rows, double *out,
                             double *lse) {
    if (B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Dk <= 0 || Dv <= 0 || P <= 0 ||
        max_pages <= 0 || v_row_stride < Dv || topk_stride <= 0)
        return -1;
    const int G = Hq / Hkv;
    const long long total_rows = (long long)B * T * Hq;
    if (rows == NULL) n_rows = total_rows;

    for (int b = 0; b < B; ++b) {
        int L = seqlens[b];
        if (L < 0 || (long long)L > (long long)max_pages * P) return -2;
        int K = topk_len[b];
        if (K < 0 || K > topk_stride) return -5;
        for (int i = 0; i < K; ++i) {
            int j = topk_idx[(long long)b * topk_stride + i];
            if (j < 0 || j >= L) return -6;
            int pg = page_table[(long long)b * max_pages + j / P];
            if (pg < 0 || pg >= num_pages) return -3;
        }
    }

    int err = 0;
#pragma omp parallel
    {
        double *sig = NULL;
        long long cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (long long i = 0; i < n_rows; ++i) {
            long long r = rows ? rows[i] : i;
            if (r < 0 || r >= total_rows) {
#pragma omp atomic write
                err = -1;
                continue;
            }
            const int h = (int)(r % Hq);
            const int b = (int)(r / ((long long)Hq * T));
            const int g = h / G;
            const long long n = topk_len[b];
            const int32_t *sel = topk_idx + (long long)b * topk_stride;
            double *o = out + i * (long long)Dv;
            for (int d = 0; d < Dv; ++d) o[d] = 0.0;
            if (n <= 0) {
                lse[i] = -INFINITY;
                continue;
            }
            if (n > cap) {
                free(sig);
                cap = n;
                sig = (double *)malloc(sizeof(double) * (size_t)cap);
            }
            const uint16_t *qr = q + r * (long long)Dk;
            for (long long x = 0; x < n; ++x) {
                const int j = sel[x];
                const int pg = page_table[(long long)b * max_pages + j / P];
                const uint16_t *kr = k_pages + (((long long)pg * P + j % P) * Hkv + g) * (long long)Dk;
                double acc = 0.0;
                for (int d = 0; d < Dk; ++d) acc += bf16_to_f64(qr[d]) * bf16_to_f64(kr[d]);
                sig[x] = scale * acc;
            }
            double mu = -INFINITY;
            for (long long x = 0; x < n; ++x)
                if (sig[x] > mu) mu = sig[x];
            double Z = 0.0;
            for (long long x = 0; x < n; ++x) Z += exp(sig[x] - mu);
            for (long long x = 0; x < n; ++x) {
                const double wgt = exp(sig[x] - mu) / Z;
                const int j = sel[x];
                const int pg = page_table[(long long)b * max_pages + j / P];
                const uint16_t *vr = v_pages + (((long long)pg * P + j % P) * Hkv + g) * v_row_stride;
                for (int d = 0; d < Dv; ++d) o[d] += wgt * bf16_to_f64(vr[d]);
            }
            lse[i] = mu + log(Z);
        }
        free(sig);
    }
    return err;
}
