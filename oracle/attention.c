/*
 * Float64 CPU oracle for paged attention.  TEST INFRASTRUCTURE ONLY: nothing
 * in the product path links, loads or calls this file.
 *
 * Sources (page title, section):
 *   P1 = "03｜PagedAttention 与 KV Cache 内存系统" (llm-infra-atlas.github.io)
 *   P2 = "KV Cache：容量、布局与生命周期" (wineandchord.com)
 *   P3 = "PagedAttention 的原理是什么？它如何降低 KV Cache 的内存浪费？" (offer.aigcbaba.com)
 *   P4 = "vLLM学习笔记-显存管理之PagedAttention" (amentiraz.github.io)
 *
 * What is computed.  P1 §4 and P3 §五 state that reading the cache through a
 * block table does not change the attention result: it equals attention over
 * the contiguous logical sequence.  So the oracle is that definition written
 * out: gather the visible logical positions through the table (P1 §3 address
 * formula, P2 "Page-table 寻址"), then plain softmax attention in float64:
 *
 *     x_i = scale * sum_d q[d] * K_i[d]
 *     out = sum_i exp(x_i - max_j x_j) V_i / sum_i exp(x_i - max_j x_j)
 *
 * Pool layout read here: K and V pools, each [num_blocks][H_kv][block_size][D]
 * of f32 or bf16 bit patterns (dtype 0 / 1), or float64 (dtype 2: FP8 pages
 * dequantised by oracle/fp8.py; the query is then float64 too).  A token at logical position p of
 * a sequence lives in block table[p / B_p] at offset p mod B_p.
 * GQA mapping (P2 "物理布局" raises it, leaves it open): q-head g reads
 * kv-head g / (H_q / H_kv).
 *
 * Every function returns 0 on success or a negative error:
 *   -1 invalid argument, -2 logical block not allocated / id out of range,
 *   -3 negative physical id.
 * No blocking, fusion or reordering: one output row at a time, keys in
 * logical order, sums in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double elem(const void* base, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float*)base)[i];
    if (dtype == 2) return ((const double*)base)[i];  /* dequantised FP8 values */
    /* bf16: the upper 16 bits of an IEEE float32 */
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* P2 "Page-table 寻址": validated slot of a token position. */
int orc_physical_slot(const int32_t* table, int64_t n_entries, int64_t block_size,
                      int64_t pos, int64_t* slot) {
    if (block_size <= 0 || pos < 0) return -1;
    int64_t logical = pos / block_size, offset = pos % block_size;
    if (logical >= n_entries) return -2;
    int64_t phys = table[logical];
    if (phys < 0) return -3;
    *slot = phys * block_size + offset;
    return 0;
}

/* One output row: attention of query vector q (D values, index into `qbase`)
 * over the first `n_vis` logical positions of a sequence whose block table is
 * `table`, for kv-head h. */
static int attend_row(const void* kpool, const void* vpool, int dtype, int32_t num_blocks,
                      int32_t Bp, int32_t Hkv, int32_t D, const void* qbase, size_t q_off,
                      const int32_t* table, int32_t n_entries, int32_t h, int64_t n_vis,
                      double scale, double* out, double* x /* scratch [n_vis] */) {
    if (n_vis <= 0) return -1;
    for (int64_t i = 0; i < n_vis; ++i) {
        int64_t slot;
        int rc = orc_physical_slot(table, n_entries, Bp, i, &slot);
        if (rc) return rc;
        int64_t blk = slot / Bp, off = slot % Bp;
        if (blk >= num_blocks) return -2;
        size_t krow = (((size_t)blk * Hkv + h) * Bp + off) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += elem(qbase, dtype, q_off + d) * elem(kpool, dtype, krow + d);
        x[i] = scale * dot;
    }
    double m = x[0];
    for (int64_t i = 1; i < n_vis; ++i) if (x[i] > m) m = x[i];
    double denom = 0.0;
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t i = 0; i < n_vis; ++i) {
        double w = exp(x[i] - m);
        denom += w;
        int64_t slot;
        orc_physical_slot(table, n_entries, Bp, i, &slot);
        int64_t blk = slot / Bp, off = slot % Bp;
        size_t vrow = (((size_t)blk * Hkv + h) * Bp + off) * D;
        for (int32_t d = 0; d < D; ++d) out[d] += w * elem(vpool, dtype, vrow + d);
    }
    for (int32_t d = 0; d < D; ++d) out[d] /= denom;
    return 0;
}

/*
 * Decode (P1 §4 pseudo-kernel semantics): one query token per sequence, at the
 * last position; it attends to all context_lens[s] tokens (positions
 * 0..n-1, the new token included).  q: [B][H_q][D]; out: [B][H_q][D] f64.
 * rows (optional): list of (s, g) pairs to compute; NULL computes all, and
 * out then holds B*H_q rows; otherwise out holds n_rows rows in list order.
 */
int orc_decode(const void* kpool, const void* vpool, int dtype, int32_t num_blocks, int32_t Bp,
               int32_t Hkv, int32_t D, const void* q, int32_t Hq, const int32_t* tables,
               int32_t max_blocks, const int32_t* context_lens, int32_t B, double scale,
               const int32_t* rows, int32_t n_rows, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Bp <= 0 || B < 0) return -1;
    int32_t G = Hq / Hkv;
    int64_t total = rows ? n_rows : (int64_t)B * Hq;
    int64_t maxn = 0;
    for (int32_t s = 0; s < B; ++s) if (context_lens[s] > maxn) maxn = context_lens[s];
    int err = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int32_t s = rows ? rows[2 * r] : (int32_t)(r / Hq);
            int32_t g = rows ? rows[2 * r + 1] : (int32_t)(r % Hq);
            int rc = attend_row(kpool, vpool, dtype, num_blocks, Bp, Hkv, D, q,
                                ((size_t)s * Hq + g) * D, tables + (size_t)s * max_blocks,
                                max_blocks, g / G, context_lens[s], scale, out + (size_t)r * D, x);
            if (rc) {
#pragma omp atomic write
                err = rc;
            }
        }
        free(x);
    }
    return err;
}

/*
 * The same decode over the contiguous cache layout of P4 §"传统策略及其缺陷"
 * (cache_k[max_batch][max_seq][n_kv_heads][head_dim]), with identical loop
 * and summation order, so its result must equal orc_decode bit for bit.
 */
int orc_decode_contiguous(const void* kcache, const void* vcache, int dtype, int32_t max_seq,
                          int32_t Hkv, int32_t D, const void* q, int32_t Hq,
                          const int32_t* context_lens, int32_t B, double scale, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int32_t G = Hq / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(max_seq > 0 ? max_seq : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < (int64_t)B * Hq; ++r) {
            int32_t s = (int32_t)(r / Hq), g = (int32_t)(r % Hq), h = g / G;
            int64_t n = context_lens[s];
            double* o = out + (size_t)r * D;
            size_t qo = ((size_t)s * Hq + g) * D;
            if (n <= 0 || n > max_seq) {
#pragma omp atomic write
                err = -1;
                continue;
            }
            for (int64_t i = 0; i < n; ++i) {
                size_t krow = (((size_t)s * max_seq + i) * Hkv + h) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += elem(q, dtype, qo + d) * elem(kcache, dtype, krow + d);
                x[i] = scale * dot;
            }
            double m = x[0];
            for (int64_t i = 1; i < n; ++i) if (x[i] > m) m = x[i];
            double denom = 0.0;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                double w = exp(x[i] - m);
                denom += w;
                size_t vrow = (((size_t)s * max_seq + i) * Hkv + h) * D;
                for (int32_t d = 0; d < D; ++d) o[d] += w * elem(vcache, dtype, vrow + d);
            }
            for (int32_t d = 0; d < D; ++d) o[d] /= denom;
        }
        free(x);
    }
    return err;
}

/*
 * Decode computed block by block with the (max, exp_sum, weighted_value)
 * state of P1 §4: the context is cut into partitions of `part_tokens`
 * positions; each partition yields m_p = max x, l_p = sum exp(x - m_p),
 * a_p = sum exp(x - m_p) V; partitions are then merged:
 *   M = max m_p, L = sum l_p exp(m_p - M), out = sum a_p exp(m_p - M) / L.
 * Used to pin that the split-KV combination reaches the unsplit result.
 */
int orc_decode_split(const void* kpool, const void* vpool, int dtype, int32_t num_blocks,
                     int32_t Bp, int32_t Hkv, int32_t D, const void* q, int32_t Hq,
                     const int32_t* tables, int32_t max_blocks, const int32_t* context_lens,
                     int32_t B, double scale, int32_t part_tokens, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || part_tokens <= 0) return -1;
    int32_t G = Hq / Hkv;
    int err = 0;
    for (int64_t r = 0; r < (int64_t)B * Hq && !err; ++r) {
        int32_t s = (int32_t)(r / Hq), g = (int32_t)(r % Hq), h = g / G;
        int64_t n = context_lens[s];
        const int32_t* table = tables + (size_t)s * max_blocks;
        size_t qo = ((size_t)s * Hq + g) * D;
        int64_t nparts = (n + part_tokens - 1) / part_tokens;
        double* pm = (double*)malloc(sizeof(double) * nparts);
        double* pl = (double*)malloc(sizeof(double) * nparts);
        double* pa = (double*)calloc((size_t)nparts * D, sizeof(double));
        double* x = (double*)malloc(sizeof(double) * part_tokens);
        for (int64_t p = 0; p < nparts && !err; ++p) {
            int64_t lo = p * part_tokens, hi = lo + part_tokens < n ? lo + part_tokens : n;
            for (int64_t i = lo; i < hi; ++i) {
                int64_t slot;
                int rc = orc_physical_slot(table, max_blocks, Bp, i, &slot);
                if (rc) { err = rc; break; }
                size_t krow = (((size_t)(slot / Bp) * Hkv + h) * Bp + slot % Bp) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += elem(q, dtype, qo + d) * elem(kpool, dtype, krow + d);
                x[i - lo] = scale * dot;
            }
            if (err) break;
            double m = x[0];
            for (int64_t i = 1; i < hi - lo; ++i) if (x[i] > m) m = x[i];
            double l = 0.0;
            for (int64_t i = lo; i < hi; ++i) {
                double w = exp(x[i - lo] - m);
                l += w;
                int64_t slot;
                orc_physical_slot(table, max_blocks, Bp, i, &slot);
                size_t vrow = (((size_t)(slot / Bp) * Hkv + h) * Bp + slot % Bp) * D;
                for (int32_t d = 0; d < D; ++d) pa[p * D + d] += w * elem(vpool, dtype, vrow + d);
            }
            pm[p] = m;
            pl[p] = l;
        }
        if (!err) {
            double M = pm[0];
            for (int64_t p = 1; p < nparts; ++p) if (pm[p] > M) M = pm[p];
            double L = 0.0;
            double* o = out + (size_t)r * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t p = 0; p < nparts; ++p) {
                double c = exp(pm[p] - M);
                L += pl[p] * c;
                for (int32_t d = 0; d < D; ++d) o[d] += pa[p * D + d] * c;
            }
            for (int32_t d = 0; d < D; ++d) o[d] /= L;
        }
        free(pm); free(pl); free(pa); free(x);
    }
    return err;
}

/*
 * Chunked prefill (P1 §4: a prefill kernel reads the same paged table).
 * Sequence s has new query tokens q[cu_seqlens_q[s] .. cu_seqlens_q[s+1]) and
 * context_lens[s] tokens in the cache including those new ones; new token i
 * sits at absolute position context_lens[s] - n_new + i.  With `causal` it sees
 * positions 0..its own (inclusive); otherwise all context_lens[s] positions.
 * q/out rows are [token][H_q][D].  rows (optional): (token, q-head) pairs.
 */
int orc_prefill(const void* kpool, const void* vpool, int dtype, int32_t num_blocks, int32_t Bp,
                int32_t Hkv, int32_t D, const void* q, int32_t Hq, const int32_t* cu_seqlens_q,
                const int32_t* context_lens, const int32_t* tables, int32_t max_blocks, int32_t B,
                double scale, int32_t causal, const int32_t* rows, int32_t n_rows, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || B <= 0) return -1;
    int32_t G = Hq / Hkv;
    int64_t T = cu_seqlens_q[B];
    int64_t total = rows ? n_rows : T * Hq;
    int64_t maxn = 0;
    for (int32_t s = 0; s < B; ++s) if (context_lens[s] > maxn) maxn = context_lens[s];
    int err = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int64_t t = rows ? rows[2 * r] : r / Hq;
            int32_t g = rows ? rows[2 * r + 1] : (int32_t)(r % Hq);
            int32_t s = 0;
            while (s + 1 < B && cu_seqlens_q[s + 1] <= t) ++s;
            int64_t n_new = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
            int64_t i = t - cu_seqlens_q[s];
            int64_t pos = context_lens[s] - n_new + i;
            int64_t n_vis = causal ? pos + 1 : context_lens[s];
            int rc = (pos < 0) ? -1
                     : attend_row(kpool, vpool, dtype, num_blocks, Bp, Hkv, D, q,
                                  ((size_t)t * Hq + g) * D, tables + (size_t)s * max_blocks,
                                  max_blocks, g / G, n_vis, scale, out + (size_t)r * D, x);
            if (rc) {
#pragma omp atomic write
                err = rc;
            }
        }
        free(x);
    }
    return err;
}

/*
 * Sliding-window decode ("03｜PagedAttention 与 KV Cache 内存系统" §1.1 and §7:
 * a sliding-window layer only uses the tokens inside its window; the window of
 * the token at position p is [p - w + 1, p]).  The query is the token at
 * position n - 1 (n = context_lens[s]), so it attends to positions
 * max(0, n - window) .. n - 1 through the block table; window <= 0 means no
 * window (all n positions, as orc_decode).  Same arguments and layout as
 * orc_decode plus `window`.
 */
int orc_decode_window(const void* kpool, const void* vpool, int dtype, int32_t num_blocks,
                      int32_t Bp, int32_t Hkv, int32_t D, const void* q, int32_t Hq,
                      const int32_t* tables, int32_t max_blocks, const int32_t* context_lens,
                      int32_t B, int32_t window, double scale, const int32_t* rows,
                      int32_t n_rows, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Bp <= 0 || B < 0) return -1;
    int32_t G = Hq / Hkv;
    int64_t total = rows ? n_rows : (int64_t)B * Hq;
    int64_t maxn = 0;
    for (int32_t s = 0; s < B; ++s) if (context_lens[s] > maxn) maxn = context_lens[s];
    int err = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int32_t s = rows ? rows[2 * r] : (int32_t)(r / Hq);
            int32_t g = rows ? rows[2 * r + 1] : (int32_t)(r % Hq);
            int32_t h = g / G;
            int64_t n = context_lens[s];
            int64_t lo = (window > 0 && n > window) ? n - window : 0;
            const int32_t* table = tables + (size_t)s * max_blocks;
            size_t q_off = ((size_t)s * Hq + g) * D;
            double* o = out + (size_t)r * D;
            int rc = 0;
            if (n <= 0) rc = -1;
            /* scores of the visible positions lo .. n-1 */
            for (int64_t i = lo; i < n && !rc; ++i) {
                int64_t slot;
                rc = orc_physical_slot(table, max_blocks, Bp, i, &slot);
                if (rc) break;
                int64_t blk = slot / Bp, off = slot % Bp;
                if (blk >= num_blocks) { rc = -2; break; }
                size_t krow = (((size_t)blk * Hkv + h) * Bp + off) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += elem(q, dtype, q_off + d) * elem(kpool, dtype, krow + d);
                x[i - lo] = scale * dot;
            }
            if (!rc) {
                /* softmax over the window, then the weighted sum of V */
                double m = x[0];
                for (int64_t i = 1; i < n - lo; ++i) if (x[i] > m) m = x[i];
                double denom = 0.0;
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t i = lo; i < n; ++i) {
                    double w = exp(x[i - lo] - m);
                    denom += w;
                    int64_t slot;
                    orc_physical_slot(table, max_blocks, Bp, i, &slot);
                    int64_t blk = slot / Bp, off = slot % Bp;
                    size_t vrow = (((size_t)blk * Hkv + h) * Bp + off) * D;
                    for (int32_t d = 0; d < D; ++d) o[d] += w * elem(vpool, dtype, vrow + d);
                }
                for (int32_t d = 0; d < D; ++d) o[d] /= denom;
            } else {
#pragma omp atomic write
                err = rc;
            }
        }
        free(x);
    }
    return err;
}
