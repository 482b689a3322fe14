/*
 * fa_oracle.c -- the CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * this library.  It shares no code, header or constant with the CUDA library: it is a
 * plain, slow, obviously correct restatement of what exact attention computes, in
 * fp64, with the score row materialised and a two-pass softmax.
 *
 * What it follows (page titles and sections of the source pages):
 *  - "flash-attention-v100", section "How to use FlashAttention": the operation is
 *    softmax(Q @ K^T * softmax_scale) @ V over tensors laid out
 *    (batch, seqlen, nheads, headdim); K/V may carry fewer heads than Q, the number of
 *    Q heads being a multiple of it, and Q head h reads K/V head h / (Hq / Hkv)
 *    (the 6-over-2 heads example in the flash_attn_func docstring).
 *  - same page, "Changelog", "2.1: Change behavior of causal flag": the causal mask is
 *    aligned to the bottom-right corner, so key j is kept for query i iff
 *    j <= i + Sk - Sq; a row whose mask is all zero produces a zero output.
 *  - same page, "Changelog", "2.2: Optimize for inference" and the search snippets on
 *    Flash-Decoding (page "flash attention-2 github", steps 1-3): the KV cache is cut
 *    into chunks, attention is taken per chunk together with one extra scalar per row
 *    and chunk (the log of the sum of exponentials), and a separate step merges them.
 *    The merge is the log-sum-exp identity over a partition of the key set, written
 *    out in fa_oracle_combine below.
 *  - same page, "How to use FlashAttention" (flash_attn_with_kvcache, block_table) and
 *    "Changelog", "2.5: Paged KV cache": with a block table, key j of sequence b lives
 *    in page block_table[b][j / page_size] at row j % page_size of a
 *    [num_pages, page_size, Hkv, D] cache.
 *  - same page, "How to use FlashAttention" (flash_attn_func, window_size) and
 *    "Changelog", "2.3: Local (i.e., sliding window) attention": with a window
 *    (left, right), query i attends only to keys j with
 *    i + Sk - Sq - left <= j <= i + Sk - Sq + right; -1 means unbounded on that side.
 *    With the causal flag the right bound is at most i + Sk - Sq (the plainest reading
 *    of combining the two: both masks apply).
 *
 * Readings where the pages are silent: the per-row log-sum-exp is the natural log of
 * the sum of exp over the *scaled, masked* scores; a row with no visible key has
 * output 0 and log-sum-exp -inf; the decode query sees keys [0, kv_len_b).
 *
 * Inputs are read as stored (bf16, fp16, fp32 or fp64) and widened exactly to double;
 * every product, sum, exp and log is taken in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_F32 = 2, ORC_F64 = 3 };

/* IEEE 754 binary16 -> double, from the format's definition (1 sign bit, 5 exponent
 * bits with bias 15, 10 fraction bits; exponent 0 is subnormal, 31 is inf/nan). */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);
    } else if (e == 31) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(f + 1024), e - 25);
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load_elem(const void *base, int dtype, size_t idx) {
    switch (dtype) {
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    case ORC_FP16: return half_bits_to_double(((const uint16_t *)base)[idx]);
    case ORC_F32: return (double)((const float *)base)[idx];
    default: return ((const double *)base)[idx];
    }
}

/*
 * Attention of one query row over the keys j0 <= j < j1 of one K/V head.
 *   q_off      element offset of q[0]
 *   kv_off     element offset of k[j = 0][0] (same for v)
 *   kv_stride  elements between key j and key j + 1
 * Scores s_j = scale * <q, k_j> are materialised in s_buf, then the two-pass softmax:
 * m = max_j s_j, l = sum_j exp(s_j - m), P_j = exp(s_j - m) / l,
 * o = sum_j P_j v_j, lse = m + ln l.  An empty key range gives o = 0, lse = -inf.
 */
static void attend_row(const void *q, const void *k, const void *v, int dtype, size_t q_off,
                       size_t kv_off, size_t kv_stride, int D, long j0, long j1, double scale,
                       double *s_buf, double *o, double *lse) {
    if (j1 <= j0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    long n = j1 - j0;
    for (long t = 0; t < n; ++t) {
        size_t kbase = kv_off + (size_t)(j0 + t) * kv_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load_elem(q, dtype, q_off + d) * load_elem(k, dtype, kbase + d);
        s_buf[t] = scale * dot;
    }
    double m = s_buf[0];
    for (long t = 1; t < n; ++t)
        if (s_buf[t] > m) m = s_buf[t];
    double l = 0.0;
    for (long t = 0; t < n; ++t) l += exp(s_buf[t] - m);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (long t = 0; t < n; ++t) {
        double p = exp(s_buf[t] - m) / l;
        size_t vbase = kv_off + (size_t)(j0 + t) * kv_stride;
        for (int d = 0; d < D; ++d) o[d] += p * load_elem(v, dtype, vbase + d);
    }
    *lse = m + log(l);
}

/* ------------------------------------------------------------------ thread pool -- */

typedef struct {
    const void *q, *k, *v;
    int dtype;
    long B, Sq, Sk, Hq, Hkv, D;
    double scale;
    int causal;
    long win_left, win_right; /* sliding window, -1 = unbounded */
    const int64_t *rows; /* (b, h, i) triples, or NULL for every row */
    const int32_t *kv_lens; /* decode mode: per-sequence key counts, else NULL */
    long n_items;
    double *o, *lse;
    int nthreads;
} fwd_job;

typedef struct {
    const fwd_job *job;
    int tid;
    int err;
} fwd_worker;

static void decode_one(const fwd_job *J, long item, double *s_buf) {
    /* item enumerates (b, h); the cache is [B, Smax = Sk, Hkv, D], q is [B, Hq, D] */
    long h = item % J->Hq;
    long b = item / J->Hq;
    long hk = h / (J->Hq / J->Hkv);
    size_t q_off = ((size_t)b * J->Hq + h) * J->D;
    size_t kv_off = (((size_t)b * J->Sk) * J->Hkv + hk) * J->D;
    attend_row(J->q, J->k, J->v, J->dtype, q_off, kv_off, (size_t)J->Hkv * J->D, (int)J->D, 0,
               J->kv_lens[b], J->scale, s_buf, J->o + (size_t)item * J->D, J->lse + item);
}

static void fwd_one(const fwd_job *J, long item, double *s_buf) {
    long b, h, i;
    double *o;
    double *lse;
    if (J->rows) {
        b = J->rows[3 * item + 0];
        h = J->rows[3 * item + 1];
        i = J->rows[3 * item + 2];
        o = J->o + (size_t)item * J->D;
        lse = J->lse + item;
    } else {
        /* item enumerates (b, h, i) with i fastest */
        i = item % J->Sq;
        h = (item / J->Sq) % J->Hq;
        b = item / (J->Sq * J->Hq);
        o = J->o + (((size_t)b * J->Sq + i) * J->Hq + h) * J->D;
        lse = J->lse + ((size_t)b * J->Hq + h) * J->Sq + i;
    }
    long g = J->Hq / J->Hkv;
    long hk = h / g; /* grouped-query head map */
    size_t q_off = (((size_t)b * J->Sq + i) * J->Hq + h) * J->D;
    size_t kv_off = (((size_t)b * J->Sk) * J->Hkv + hk) * J->D;
    size_t kv_stride = (size_t)J->Hkv * J->D;
    long j0 = 0, j1 = J->Sk;
    if (J->causal) {
        long lim = i + J->Sk - J->Sq + 1; /* bottom-right aligned: j <= i + Sk - Sq */
        if (lim < j1) j1 = lim;
    }
    if (J->win_right >= 0) {
        long lim = i + J->Sk - J->Sq + J->win_right + 1;
        if (lim < j1) j1 = lim;
    }
    if (J->win_left >= 0) {
        long lim = i + J->Sk - J->Sq - J->win_left;
        if (lim > j0) j0 = lim;
    }
    attend_row(J->q, J->k, J->v, J->dtype, q_off, kv_off, kv_stride, (int)J->D, j0, j1, J->scale,
               s_buf, o, lse);
}

static void *fwd_worker_main(void *arg) {
    fwd_worker *w = (fwd_worker *)arg;
    const fwd_job *J = w->job;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
    if (!s_buf) {
        w->err = 1;
        return NULL;
    }
    for (long it = w->tid; it < J->n_items; it += J->nthreads) {
        if (J->kv_lens)
            decode_one(J, it, s_buf);
        else
            fwd_one(J, it, s_buf);
    }
    free(s_buf);
    return NULL;
}

static int run_pool(fwd_job *J) {
    int nt = J->nthreads;
    if (nt < 1) nt = 1;
    if (nt > J->n_items) nt = (int)(J->n_items > 0 ? J->n_items : 1);
    J->nthreads = nt;
    fwd_worker *ws = (fwd_worker *)calloc((size_t)nt, sizeof(fwd_worker));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!ws || !th) {
        free(ws);
        free(th);
        return 3;
    }
    int err = 0;
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        ws[t].job = J;
        ws[t].tid = t;
        if (t == 0) continue;
        if (pthread_create(&th[t], NULL, fwd_worker_main, &ws[t]) != 0) {
            err = 3;
            break;
        }
        started = t;
    }
    if (!err) fwd_worker_main(&ws[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nt && !err; ++t)
        if (ws[t].err) err = 3;
    free(ws);
    free(th);
    return err;
}

/* ------------------------------------------------------------------ public API --- */

/*
 * Exact attention forward for [B, S, H, D] tensors (page "flash-attention-v100",
 * "How to use FlashAttention", flash_attn_func), optionally restricted to a sliding
 * window (win_left / win_right, -1 = unbounded).
 *   rows == NULL: every row; o is [B, Sq, Hq, D], lse is [B, Hq, Sq].
 *   rows != NULL: n_rows (b, h, i) triples; o is [n_rows, D], lse is [n_rows].
 * Returns 0 on success, 2 on a bad argument, 3 when out of host memory.
 */
int fa_oracle_fwd(const void *q, const void *k, const void *v, int dtype, long B, long Sq,
                  long Sk, long Hq, long Hkv, long D, double scale, int causal, long win_left,
                  long win_right, const int64_t *rows, long n_rows, double *o, double *lse,
                  int nthreads) {
    if (!q || !k || !v || !o || !lse) return 2;
    if (B < 0 || Sq < 0 || Sk < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return 2;
    if (Hq % Hkv != 0) return 2;
    if (dtype < ORC_BF16 || dtype > ORC_F64) return 2;
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.k = k;
    J.v = v;
    J.dtype = dtype;
    J.B = B;
    J.Sq = Sq;
    J.Sk = Sk;
    J.Hq = Hq;
    J.Hkv = Hkv;
    J.D = D;
    J.scale = scale;
    J.causal = causal;
    J.win_left = win_left;
    J.win_right = win_right;
    J.o = o;
    J.lse = lse;
    J.nthreads = nthreads;
    if (rows) {
        for (long r = 0; r < n_rows; ++r) {
            if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 ||
                rows[3 * r + 1] >= Hq || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Sq)
                return 2;
        }
        J.rows = rows;
        J.n_items = n_rows;
    } else {
        J.n_items = B * Hq * Sq;
    }
    if (J.n_items == 0) return 0;
    return run_pool(&J);
}

/*
 * Attention of the query of (b, h) over the key range [j0, j1) of a KV cache laid out
 * [B, Smax, Hkv, D]: one split's partial output and its log-sum-exp (page "flash
 * attention-2 github", Flash-Decoding step 2).  q is [B, Hq, D] (one query token).
 */
int fa_oracle_partial(const void *q, const void *k_cache, const void *v_cache, int dtype,
                      long B, long Hq, long Hkv, long D, long Smax, long b, long h, long j0,
                      long j1, double scale, double *o, double *lse) {
    if (!q || !k_cache || !v_cache || !o || !lse) return 2;
    if (Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 2;
    if (b < 0 || b >= B || h < 0 || h >= Hq) return 2;
    if (j0 < 0 || j1 > Smax) return 2;
    long hk = h / (Hq / Hkv);
    size_t q_off = ((size_t)b * Hq + h) * D;
    size_t kv_off = (((size_t)b * Smax) * Hkv + hk) * D;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(j1 > j0 ? j1 - j0 : 1));
    if (!s_buf) return 3;
    /* attend_row indexes keys from 0; shift the base so key j0 sits at index j0 */
    attend_row(q, k_cache, v_cache, dtype, q_off, kv_off, (size_t)Hkv * D, (int)D, j0, j1, scale,
               s_buf, o, lse);
    free(s_buf);
    return 0;
}

/*
 * Single-token decode over a KV cache with per-sequence lengths: the query of
 * sequence b attends to keys [0, kv_lens[b]) (page "flash-attention-v100",
 * flash_attn_with_kvcache, cache_seqlens).  q is [B, Hq, D]; o is [B, Hq, D];
 * lse is [B, Hq].  This is the definition, not the split algorithm.
 */
int fa_oracle_decode(const void *q, const void *k_cache, const void *v_cache, int dtype,
                     const int32_t *kv_lens, long B, long Hq, long Hkv, long D, long Smax,
                     double scale, double *o, double *lse, int nthreads) {
    if (!q || !k_cache || !v_cache || !kv_lens || !o || !lse) return 2;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Smax < 0 || Hq % Hkv != 0) return 2;
    if (dtype < ORC_BF16 || dtype > ORC_F64) return 2;
    for (long b = 0; b < B; ++b)
        if (kv_lens[b] < 0 || kv_lens[b] > Smax) return 2;
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.k = k_cache;
    J.v = v_cache;
    J.dtype = dtype;
    J.B = B;
    J.Sq = 1;
    J.Sk = Smax;
    J.Hq = Hq;
    J.Hkv = Hkv;
    J.D = D;
    J.scale = scale;
    J.kv_lens = kv_lens;
    J.o = o;
    J.lse = lse;
    J.nthreads = nthreads;
    J.n_items = B * Hq;
    if (J.n_items == 0) return 0;
    return run_pool(&J);
}

/*
 * Merge n partial results over disjoint key sets (Flash-Decoding step 3): with
 * lse = ln sum_s exp(lse_s), the merged output is sum_s exp(lse_s - lse) * o_s.
 * Partials with lse_s = -inf carry no keys and weigh 0; if all are -inf the result is
 * o = 0, lse = -inf.  o_parts is [n, D].
 */
int fa_oracle_combine(const double *o_parts, const double *lse_parts, long n, long D, double *o,
                      double *lse) {
    if (!o || !lse || D <= 0 || n < 0) return 2;
    double mx = -INFINITY;
    for (long s = 0; s < n; ++s)
        if (lse_parts[s] > mx) mx = lse_parts[s];
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    if (mx == -INFINITY) {
        *lse = -INFINITY;
        return 0;
    }
    double sum = 0.0;
    for (long s = 0; s < n; ++s) sum += exp(lse_parts[s] - mx);
    double total = mx + log(sum);
    for (long s = 0; s < n; ++s) {
        double w = exp(lse_parts[s] - total);
        for (long d = 0; d < D; ++d) o[d] += w * o_parts[s * D + d];
    }
    *lse = total;
    return 0;
}

/*
 * Single-token decode over a paged KV cache (page "flash-attention-v100",
 * flash_attn_with_kvcache with block_table; "Changelog", "2.5: Paged KV cache"):
 * k_pages / v_pages are [num_pages, page_size, Hkv, D]; block_table is
 * [B, max_pages] (host int32); key j of sequence b is row j % page_size of page
 * block_table[b][j / page_size].  The keys of each sequence are first gathered into a
 * contiguous fp64 buffer in that order, then the decode definition is applied.
 */
int fa_oracle_decode_paged(const void *q, const void *k_pages, const void *v_pages, int dtype,
                           const int32_t *block_table, const int32_t *kv_lens, long B, long Hq,
                           long Hkv, long D, long num_pages, long page_size, long max_pages,
                           double scale, double *o, double *lse, int nthreads) {
    if (!q || !k_pages || !v_pages || !block_table || !kv_lens || !o || !lse) return 2;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || max_pages <= 0) return 2;
    if (Hq % Hkv != 0) return 2;
    const long smax = page_size * max_pages;
    for (long b = 0; b < B; ++b) {
        if (kv_lens[b] < 0 || kv_lens[b] > smax) return 2;
        for (long t = 0; t * page_size < kv_lens[b]; ++t) {
            const long pg = block_table[b * max_pages + t];
            if (pg < 0 || pg >= num_pages) return 2;
        }
    }
    const size_t row = (size_t)Hkv * D;
    double *kc = (double *)malloc(sizeof(double) * (size_t)B * smax * row);
    double *vc = (double *)malloc(sizeof(double) * (size_t)B * smax * row);
    double *qd = (double *)malloc(sizeof(double) * (size_t)B * Hq * D);
    if (!kc || !vc || !qd) {
        free(kc);
        free(vc);
        free(qd);
        return 3;
    }
    for (size_t n = 0; n < (size_t)B * Hq * D; ++n) qd[n] = load_elem(q, dtype, n);
    for (long b = 0; b < B; ++b) {
        for (long j = 0; j < kv_lens[b]; ++j) {
            const long pg = block_table[b * max_pages + j / page_size];
            const size_t src = ((size_t)pg * page_size + (size_t)(j % page_size)) * row;
            const size_t dst = ((size_t)b * smax + (size_t)j) * row;
            for (size_t e = 0; e < row; ++e) {
                kc[dst + e] = load_elem(k_pages, dtype, src + e);
                vc[dst + e] = load_elem(v_pages, dtype, src + e);
            }
        }
    }
    int rc = fa_oracle_decode(qd, kc, vc, ORC_F64, kv_lens, B, Hq, Hkv, D, smax, scale, o, lse,
                              nthreads);
    free(kc);
    free(vc);
    free(qd);
    return rc;
}
