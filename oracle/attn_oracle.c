/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for scaled-dot-product
 * attention as the kernels of this library compute it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links or calls this file;
 * only the tests, the package smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, per (sequence or prompt b, query head h, query i), with
 * every input value widened exactly to double:
 *
 *   g      = h / (Hq / Hkv)                          GQA: contiguous head groups
 *   keep(j)= j < L  and (causal -> j <= pos_i)
 *                   and (window > 0 -> pos_i - j < window        if causal
 *                                      |pos_i - j| < window      otherwise)
 *   s_j    = scale * sum_d q[i,h,d] * k[j,g,d]
 *   s_j    = c * tanh(s_j / c)                       only when softcap c > 0
 *   m      = max_{keep} s_j
 *   p_j    = exp(s_j - m)                            (0 where !keep)
 *   o[i,h] = sum_j p_j v[j,g,:] / sum_j p_j,   lse = m + log(sum_j p_j)
 *
 * Sources (pages on the subject):
 *   - doppler src/gpu/kernels/attention.js, createAttentionUniformBuffer:
 *     the parameter block (numHeads, numKVHeads, headDim, kvLen, seqLen, scale,
 *     causal, startPos, attnSoftcap with 0 = disabled, slidingWindow with
 *     0 = disabled, kvStart, pageSize, kvLayout contiguous/ring/paged).
 *   - doppler src/inference/pipelines/text/attention/run.js,
 *     runLayerAttentionGPU: decode appends the new token's K/V before
 *     attention, so the query position is kvLen-1; the sliding-window clamp
 *     kvLen = min(kvLen, W), kvStart = total - kvLen keeps the W most recent
 *     keys including the query's own; scale = 1/sqrt(query_pre_attn_scalar)
 *     or 1/sqrt(headDim).
 *   - doppler attention.js, executeAttentionTieredQuant: an int8 K/V tier with
 *     separate K and V scale buffers (granularity: one f16 scale per
 *     (token, kv-head); value = code * scale).
 *   - rullama src/backend/dispatch/attention.rs, vision_attention_chained:
 *     vision attention is the same computation without the causal mask.
 *
 * Decode caches:
 *   contiguous: k[b][t][g][d],      scales [b][g][t]   (t < cap)
 *   paged:      k[page][r][g][d],   scales [page][g][r]
 *               page = page_table[b][t / P], r = t % P
 *   (attention.js passes the page table and pageSize to the paged decode
 *    variant; logical token t lives in row t % P of page table[t / P].)
 *
 * Parity pins: the tests check this file against closed forms, a brute-force
 * library softmax on the full score matrix, mask enumeration, and layout
 * equivalences; none of them calls back into this code to produce an
 * expected value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE-754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* keep(j) for a query at position pos over keys 0..L-1 */
static int oracle_keep(long pos, long j, long L, int causal, int window)
{
    if (j < 0 || j >= L) return 0;
    if (causal && j > pos) return 0;
    if (window > 0) {
        long dist = pos - j;
        if (!causal && dist < 0) dist = -dist;
        if (dist >= window) return 0;
    }
    return 1;
}

/* Attention of one query row against L key/value rows (all double).
 * Two passes: the max of the kept logits, then the weighted sums. */
static void oracle_attend(const double* q, const double* K, const double* V,
                          long L, int D, long pos, int causal, int window,
                          double softcap, double scale, double* o, double* lse)
{
    double* s = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
    double m = -INFINITY;
    for (long j = 0; j < L; ++j) {
        if (!oracle_keep(pos, j, L, causal, window)) { s[j] = -INFINITY; continue; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * K[j * D + d];
        double x = scale * dot;
        if (softcap > 0.0) x = softcap * tanh(x / softcap);
        s[j] = x;
        if (x > m) m = x;
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) {             /* nothing kept: zero output, lse = -inf */
        *lse = -INFINITY;
        free(s);
        return;
    }
    double l = 0.0;
    for (long j = 0; j < L; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) o[d] += p * V[j * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
    free(s);
}

/* One query element: q is f16 bits, or binary32 values when q_f32 (the f32-Q
 * variant: attention.js executeAttentionTieredQuant takes f32 Q only; a float
 * widens to double exactly). */
static double oracle_q_value(const void* q, int q_f32, long idx)
{
    if (q_f32) return (double)((const float*)q)[idx];
    return oracle_f16_to_double(((const uint16_t*)q)[idx]);
}

/* One cache element (token t of sequence b, kv head g, dim d) as double. */
static double oracle_cache_value(const void* cache, const uint16_t* scales, int is_int8,
                                 const int32_t* page_table, int P, int max_pages, long cap,
                                 long n_pages, int b, long t, int g, int d, int Hkv, int D)
{
    long row_base, scale_idx;
    if (page_table) {
        long page = page_table[(long)b * max_pages + t / P];
        long r = t % P;
        if (page < 0 || page >= n_pages) return NAN;     /* invalid page id */
        row_base = ((page * P + r) * Hkv + g) * (long)D;
        scale_idx = (page * Hkv + g) * (long)P + r;
    } else {
        row_base = (((long)b * cap + t) * Hkv + g) * (long)D;
        scale_idx = ((long)b * Hkv + g) * cap + t;
    }
    if (is_int8) {
        double code = (double)((const int8_t*)cache)[row_base + d];
        return code * oracle_f16_to_double(scales[scale_idx]);
    }
    return oracle_f16_to_double(((const uint16_t*)cache)[row_base + d]);
}

/*
 * Decode: one new query per sequence, at position kv_len[b]-1.  q [B][Hq][D]:
 * f16 bits, or binary32 when q_f32.
 * rows: n_rows (b, h) pairs to evaluate (rows_b/rows_h), or n_rows < 0 for all
 * B*Hq in (b, h) row-major order.  out: [n][D], lse: [n].
 * ring > 0: the cache is a ring of `ring` slots per sequence (doppler run.js,
 * runLayerAttentionGPU: a SlidingWindowKVCache selects kvLayout 'ring' and
 * kvStart = totalSeqLen - kvLen): logical token t lives in slot t % ring of the
 * contiguous [B][ring][Hkv][D] layout, kv_len is the logical length (not
 * clamped), and the kept keys are the last min(kv_len, ring, window) tokens.
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_decode(const void* q, int q_f32, const void* k, const void* v, int kv_int8,
                  const uint16_t* k_scales, const uint16_t* v_scales,
                  const int32_t* kv_len, const int32_t* page_table,
                  int page_size, int max_pages, long cap, long n_pages,
                  int B, int Hq, int Hkv, int D, int window, double softcap, double scale,
                  int n_rows, const int32_t* rows_b, const int32_t* rows_h,
                  double* out, double* lse, int n_threads, int ring)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    if (page_table && page_size <= 0) return -1;
    if (ring > 0 && (page_table || ring != cap)) return -1;
    int G = Hq / Hkv;
    long n = n_rows < 0 ? (long)B * Hq : n_rows;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long r = 0; r < n; ++r) {
        int b = n_rows < 0 ? (int)(r / Hq) : rows_b[r];
        int h = n_rows < 0 ? (int)(r % Hq) : rows_h[r];
        int g = h / G;
        long L = kv_len[b];
        long cap_b = page_table ? (long)max_pages * page_size : cap;
        if (L < 0) L = 0;
        if (ring > 0) {
            /* the kept logical keys t0 .. L-1, gathered from their slots t % ring */
            long keep = L < ring ? L : ring;
            if (window > 0 && window < keep) keep = window;
            long t0 = L - keep;
            double* qd = (double*)malloc(sizeof(double) * D);
            double* Kd = (double*)malloc(sizeof(double) * (size_t)(keep > 0 ? keep : 1) * D);
            double* Vd = (double*)malloc(sizeof(double) * (size_t)(keep > 0 ? keep : 1) * D);
            for (int d = 0; d < D; ++d)
                qd[d] = oracle_q_value(q, q_f32, ((long)b * Hq + h) * D + d);
            for (long t = 0; t < keep; ++t)
                for (int d = 0; d < D; ++d) {
                    long slot = (t0 + t) % ring;
                    Kd[t * D + d] = oracle_cache_value(k, k_scales, kv_int8, NULL, 0, 0, cap, 0, b, slot, g, d, Hkv, D);
                    Vd[t * D + d] = oracle_cache_value(v, v_scales, kv_int8, NULL, 0, 0, cap, 0, b, slot, g, d, Hkv, D);
                }
            /* every gathered key is kept: the query is the last of them */
            oracle_attend(qd, Kd, Vd, keep, D, keep - 1, 1, 0, softcap, scale, out + r * D, lse + r);
            free(qd); free(Kd); free(Vd);
            continue;
        }
        if (L > cap_b) L = cap_b;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        for (int d = 0; d < D; ++d)
            qd[d] = oracle_q_value(q, q_f32, ((long)b * Hq + h) * D + d);
        for (long t = 0; t < L; ++t)
            for (int d = 0; d < D; ++d) {
                Kd[t * D + d] = oracle_cache_value(k, k_scales, kv_int8, page_table, page_size,
                                                   max_pages, cap, n_pages, b, t, g, d, Hkv, D);
                Vd[t * D + d] = oracle_cache_value(v, v_scales, kv_int8, page_table, page_size,
                                                   max_pages, cap, n_pages, b, t, g, d, Hkv, D);
            }
        /* decode is causal at position L-1: causal masks nothing inside L */
        oracle_attend(qd, Kd, Vd, L, D, L - 1, 1, window, softcap, scale,
                      out + r * D, lse + r);
        free(qd); free(Kd); free(Vd);
    }
    return 0;
}

/*
 * Tiered decode (doppler attention.js, executeAttentionTiered and
 * executeAttentionTieredQuant: a hot tier and a cold tier read in one pass,
 * hotLayout 'ring', coldLayout 'paged' or contiguous, hotWindow, hotStart).
 * Sequence b's keys are its cold_len[b] cold tokens followed by its
 * hot_len[b] hot tokens:
 *   cold token j  at position j, read from the cold cache like oracle_decode
 *                 (contiguous [B][cold_cap][Hkv][D] or paged; f16 or int8 with
 *                 scales); cold_len is clamped to [0, capacity];
 *   hot token i   at position cold_len + i, read from the f16 ring
 *                 [B][hot_ring][Hkv][D], slot (hot_start[b] + i) mod hot_ring;
 *                 the ring holds only the newest hot_ring hot tokens.
 * The query sits at cold_len + hot_len - 1 (the newest token); a window W > 0
 * keeps the keys whose position is within W of it.  Positions can skip
 * (overwritten hot tokens), so the window is applied by position here and
 * the kept keys are then attended without further masking.
 */
int oracle_decode_tiered(const void* q, int q_f32,
                         const void* ck, const void* cv, int cold_int8,
                         const uint16_t* ck_scales, const uint16_t* cv_scales,
                         const int32_t* cold_len, const int32_t* page_table,
                         int page_size, int max_pages, long cold_cap, long n_pages,
                         const uint16_t* hk, const uint16_t* hv,
                         const int32_t* hot_len, const int32_t* hot_start, long hot_ring,
                         int B, int Hq, int Hkv, int D, int window, double softcap, double scale,
                         int n_rows, const int32_t* rows_b, const int32_t* rows_h,
                         double* out, double* lse, int n_threads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || hot_ring <= 0) return -1;
    if (page_table && page_size <= 0) return -1;
    int G = Hq / Hkv;
    long n = n_rows < 0 ? (long)B * Hq : n_rows;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long r = 0; r < n; ++r) {
        int b = n_rows < 0 ? (int)(r / Hq) : rows_b[r];
        int h = n_rows < 0 ? (int)(r % Hq) : rows_h[r];
        int g = h / G;
        long cap_b = page_table ? (long)max_pages * page_size : cold_cap;
        long Lc = cold_len[b];
        if (Lc < 0) Lc = 0;
        if (Lc > cap_b) Lc = cap_b;
        long Lh = hot_len[b];
        if (Lh < 0) Lh = 0;
        long h_first = Lh > hot_ring ? Lh - hot_ring : 0;    /* older hot tokens were overwritten */
        long qpos = Lc + Lh - 1;
        long nk = Lc + (Lh - h_first);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
        for (int d = 0; d < D; ++d)
            qd[d] = oracle_q_value(q, q_f32, ((long)b * Hq + h) * D + d);
        long kept = 0;
        for (long j = 0; j < Lc; ++j) {
            if (window > 0 && qpos - j >= window) continue;
            for (int d = 0; d < D; ++d) {
                Kd[kept * D + d] = oracle_cache_value(ck, ck_scales, cold_int8, page_table, page_size,
                                                      max_pages, cold_cap, n_pages, b, j, g, d, Hkv, D);
                Vd[kept * D + d] = oracle_cache_value(cv, cv_scales, cold_int8, page_table, page_size,
                                                      max_pages, cold_cap, n_pages, b, j, g, d, Hkv, D);
            }
            ++kept;
        }
        for (long i = h_first; i < Lh; ++i) {
            if (window > 0 && qpos - (Lc + i) >= window) continue;
            long slot = ((long)hot_start[b] + i) % hot_ring;
            if (slot < 0) slot += hot_ring;
            long row = (((long)b * hot_ring + slot) * Hkv + g) * (long)D;
            for (int d = 0; d < D; ++d) {
                Kd[kept * D + d] = oracle_f16_to_double(hk[row + d]);
                Vd[kept * D + d] = oracle_f16_to_double(hv[row + d]);
            }
            ++kept;
        }
        /* every gathered key is kept: no further mask */
        oracle_attend(qd, Kd, Vd, kept, D, kept - 1, 1, 0, softcap, scale, out + r * D, lse + r);
        free(qd); free(Kd); free(Vd);
    }
    return 0;
}

/*
 * Prefill / vision: S queries at positions 0..S-1 over the same S keys.
 * q [S][Hq][D], k/v [S][Hkv][D] (f16 bits).  rows: n_rows (i, h) pairs, or
 * n_rows < 0 for all S*Hq in (i, h) row-major order.  out: [n][D], lse: [n].
 */
int oracle_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   int S, int Hq, int Hkv, int D, int causal, int window,
                   double softcap, double scale,
                   int n_rows, const int32_t* rows_i, const int32_t* rows_h,
                   double* out, double* lse, int n_threads)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    long n = n_rows < 0 ? (long)S * Hq : n_rows;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (long r = 0; r < n; ++r) {
        int i = n_rows < 0 ? (int)(r / Hq) : rows_i[r];
        int h = n_rows < 0 ? (int)(r % Hq) : rows_h[r];
        int g = h / G;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1) * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1) * D);
        for (int d = 0; d < D; ++d)
            qd[d] = oracle_f16_to_double(q[((long)i * Hq + h) * D + d]);
        for (long j = 0; j < S; ++j)
            for (int d = 0; d < D; ++d) {
                Kd[j * D + d] = oracle_f16_to_double(k[(j * Hkv + g) * (long)D + d]);
                Vd[j * D + d] = oracle_f16_to_double(v[(j * Hkv + g) * (long)D + d]);
            }
        oracle_attend(qd, Kd, Vd, S, D, i, causal, window, softcap, scale,
                      out + r * D, lse + r);
        free(qd); free(Kd); free(Vd);
    }
    return 0;
}

/*
 * Chunked prefill / multi-token decode against a paged cache: sequence b has
 * q_len = q_start[b+1] - q_start[b] new query tokens, packed as rows
 * q_start[b] .. q_start[b+1]-1 of q [total_q][Hq][D].  Their K/V are already
 * the last q_len of the kv_len[b] cache tokens, so query i sits at position
 * kv_len[b] - q_len + i and attends causally (doppler attention.js,
 * createAttentionUniformBuffer: seqLen new tokens at startPos over kvLen keys,
 * causal, with the paged layout's page table and pageSize; decode is the
 * seqLen = 1 case).  Keys past the cache capacity max_pages*P do not exist; a
 * query whose position is negative sees no key.
 * rows: n_rows (packed query row, head) pairs, or n_rows < 0 for all
 * total_q*Hq in (row, head) row-major order.  out: [n][D], lse: [n].
 */
int oracle_prefill_paged(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* q_start, const int32_t* kv_len, const int32_t* page_table,
                         int page_size, int max_pages, long n_pages,
                         int B, int Hq, int Hkv, int D, int window, double softcap, double scale,
                         int n_rows, const int32_t* rows_r, const int32_t* rows_h,
                         double* out, double* lse, int n_threads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || page_size <= 0) return -1;
    int G = Hq / Hkv;
    long total_q = q_start[B];
    long cap = (long)max_pages * page_size;
    long n = n_rows < 0 ? total_q * Hq : n_rows;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (long r = 0; r < n; ++r) {
        long row = n_rows < 0 ? r / Hq : rows_r[r];
        int h = n_rows < 0 ? (int)(r % Hq) : rows_h[r];
        int b = 0;
        while (b + 1 < B && q_start[b + 1] <= row) ++b;      /* the sequence owning the row */
        long q_len = q_start[b + 1] - q_start[b];
        long i = row - q_start[b];
        long L = kv_len[b] < cap ? kv_len[b] : cap;
        if (L < 0) L = 0;
        long pos = (long)kv_len[b] - q_len + i;
        int g = h / G;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        for (int d = 0; d < D; ++d)
            qd[d] = oracle_f16_to_double(q[(row * Hq + h) * (long)D + d]);
        for (long t = 0; t < L; ++t)
            for (int d = 0; d < D; ++d) {
                Kd[t * D + d] = oracle_cache_value(k, NULL, 0, page_table, page_size, max_pages, cap,
                                                   n_pages, b, t, g, d, Hkv, D);
                Vd[t * D + d] = oracle_cache_value(v, NULL, 0, page_table, page_size, max_pages, cap,
                                                   n_pages, b, t, g, d, Hkv, D);
            }
        if (pos < 0) {                     /* no key at or before a negative position */
            for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
            lse[r] = -INFINITY;
        } else {
            oracle_attend(qd, Kd, Vd, L, D, pos, 1, window, softcap, scale, out + r * D, lse + r);
        }
        free(qd); free(Kd); free(Vd);
    }
    return 0;
}

/* Number of threads OpenMP would use (for reporting the CPU baseline). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
