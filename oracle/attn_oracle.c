/*
 * CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the benchmark's CPU-baseline leg and
 * the smoke check may load this library. It shares no code with the CUDA path.
 *
 * What it computes is the plain definition of scaled-dot-product attention
 * ("FlashAttention: not computing less, moving less", section 01, the formula
 * O = softmax(Q K^T / sqrt(d)) V), which the tiled online-softmax kernels reach
 * exactly in real arithmetic (same page, section 02, "professional extension":
 * online softmax equals the full-row softmax). Per query row it is written out
 * as three passes in float64:
 *   s_j = scale * <q, k_j>           for every visible key j
 *   m   = max_j s_j
 *   l   = sum_j exp(s_j - m)
 *   o   = sum_j (exp(s_j - m) / l) * v_j,   lse = m + ln(l)
 * The log-sum-exp output follows the same page's section 03 ("the forward pass
 * saves the output and log-sum-exp statistics"): natural log, of scaled scores.
 *
 * Readings where the pages are silent:
 *  - causal masks are bottom-right aligned: key j is visible to query row i of a
 *    sequence with Nq queries and Nk keys iff j <= i + (Nk - Nq);
 *  - a row with no visible key has o = 0 and lse = -inf;
 *  - query head h reads key/value head h / (Hq / Hkv).
 *
 * Paged decode ("Faster, more flexible FA4 for LLM inference", PR 1999/2104 and
 * PR 1940 sections) is the same definition with one query per sequence and every
 * cached key visible; the oracle first gathers the sequence's K/V rows through
 * the page table into contiguous arrays, then applies the row routine.
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline double bf16d(uint16_t h) {
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* One query row against the first n_vis keys of a contiguous key/value array.
 * krow(j) = k + j * kv_stride, vrow(j) = v + j * kv_stride (each d elements). */
static void attend_row(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t kv_stride,
                       int64_t n_vis, int d, double scale, double* s, double* qd, double* o, double* lse) {
    if (n_vis <= 0) {
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int c = 0; c < d; ++c) qd[c] = bf16d(q[c]);
    /* scores */
    for (int64_t j = 0; j < n_vis; ++j) {
        const uint16_t* kr = k + j * kv_stride;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qd[c] * bf16d(kr[c]);
        s[j] = scale * acc;
    }
    /* pass 1: row maximum */
    double m = s[0];
    for (int64_t j = 1; j < n_vis; ++j)
        if (s[j] > m) m = s[j];
    /* pass 2: normaliser */
    double l = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) l += exp(s[j] - m);
    /* pass 3: probabilities times values */
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        const double p = exp(s[j] - m) / l;
        const uint16_t* vr = v + j * kv_stride;
        for (int c = 0; c < d; ++c) o[c] += p * bf16d(vr[c]);
    }
    *lse = m + log(l);
}

static void attend_row_f64(const double* qd, const double* k, const double* v, int64_t kstride, int64_t vstride,
                           int64_t n, int d, int dv, double scale, double* s, double* o, double* lse);

/* ------------------------------------------------------------------ forward */

typedef struct {
    const uint16_t *q, *k, *v;
    const double *qf, *kf, *vf; /* float64 inputs (oracle_attn_fwd_f64) */
    double *o, *lse;
    int B, Hq, Hkv, Nq, Nk, d, causal;
    int dv; /* value / output width (oracle_attn_fwd_f64); d for the others */
    double scale;
    const int32_t* cu; /* host cu_seqlens or NULL */
    const int64_t* rows;  /* optional (token * Hq + head) list */
    int64_t n_rows;
    int64_t next;         /* work counter */
    int64_t max_keys;
    int status;
} fwd_job_t;

/* Sequence geometry of query token t: sequence b, row i, Nq_b, Nk_b, first key token. */
static int locate(const fwd_job_t* J, int64_t t, int64_t* i, int64_t* nq, int64_t* nk, int64_t* k0) {
    if (J->cu) {
        int lo = 0, hi = J->B; /* find b with cu[b] <= t < cu[b+1] */
        if (t < J->cu[0] || t >= J->cu[J->B]) return -1;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (J->cu[mid] <= t) lo = mid; else hi = mid;
        }
        *i = t - J->cu[lo];
        *nq = *nk = J->cu[lo + 1] - J->cu[lo];
        *k0 = J->cu[lo];
    } else {
        const int64_t b = t / J->Nq;
        if (b >= J->B) return -1;
        *i = t % J->Nq;
        *nq = J->Nq;
        *nk = J->Nk;
        *k0 = b * (int64_t)J->Nk;
    }
    return 0;
}

static void* fwd_worker(void* p) {
    fwd_job_t* J = (fwd_job_t*)p;
    const int d = J->d;
    const int G = J->Hq / J->Hkv;
    const int64_t total_tokens = J->cu ? J->cu[J->B] : (int64_t)J->B * J->Nq;
    const int64_t n_items = J->rows ? J->n_rows : total_tokens * J->Hq;
    double* s = (double*)malloc(sizeof(double) * (size_t)(J->max_keys > 0 ? J->max_keys : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !qd) {
        __atomic_store_n(&J->status, -2, __ATOMIC_RELAXED);
        free(s);
        free(qd);
        return NULL;
    }
    for (;;) {
        const int64_t it = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (it >= n_items) break;
        const int64_t row = J->rows ? J->rows[it] : it;
        const int64_t t = row / J->Hq;
        const int h = (int)(row % J->Hq);
        int64_t i, nq, nk, k0;
        if (row < 0 || locate(J, t, &i, &nq, &nk, &k0) != 0) {
            __atomic_store_n(&J->status, -3, __ATOMIC_RELAXED);
            continue;
        }
        int64_t n_vis = nk;
        if (J->causal) {
            const int64_t last = i + (nk - nq); /* last visible key index */
            n_vis = last + 1 < nk ? last + 1 : nk;
        }
        const int g = h / G;
        const int64_t kv_stride = (int64_t)J->Hkv * d;
        attend_row(J->q + (t * J->Hq + h) * d, J->k + k0 * kv_stride + (int64_t)g * d,
                   J->v + k0 * kv_stride + (int64_t)g * d, kv_stride, n_vis, d, J->scale, s, qd,
                   J->o + it * d, J->lse + it);
    }
    free(s);
    free(qd);
    return NULL;
}

static int run_threads(void* (*fn)(void*), void* job, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    pthread_t th[512];
    int ok[512];
    for (int t = 0; t < n_threads; ++t) ok[t] = pthread_create(&th[t], NULL, fn, job) == 0;
    int any = 0;
    for (int t = 0; t < n_threads; ++t)
        if (ok[t]) { pthread_join(th[t], NULL); any = 1; }
    if (!any) fn(job);
    return 0;
}

/*
 * Forward attention. q: [T, Hq, d]; k, v: [Tk, Hkv, d] (bf16 bits, d fastest).
 * Dense (cu_seqlens == NULL): T = B*Nq, Tk = B*Nk, sequence b owns rows b*Nq.. and keys b*Nk...
 * Varlen (cu_seqlens = host int32[B+1]): sequence b owns tokens [cu[b], cu[b+1]) of both q and k.
 * rows == NULL: o is [T, Hq, d], lse [T, Hq]. Otherwise only the listed rows
 * (token*Hq + head) are computed and o is [n_rows, d], lse [n_rows], in list order.
 * Returns 0, or negative on bad arguments.
 */
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o, double* lse,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, double scale, int causal,
                    const int32_t* cu_seqlens, const int64_t* rows, int64_t n_rows, int n_threads) {
    if (!q || !k || !v || !o || !lse || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0) return -1;
    fwd_job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.Nq = Nq; J.Nk = Nk; J.d = d; J.causal = causal;
    J.scale = scale; J.cu = cu_seqlens; J.rows = rows; J.n_rows = n_rows;
    if (cu_seqlens) {
        int64_t mx = 0;
        for (int b = 0; b < B; ++b) {
            const int64_t L = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
            if (L < 0) return -1;
            if (L > mx) mx = L;
        }
        J.max_keys = mx;
    } else {
        if (Nq < 0 || Nk < 0) return -1;
        J.max_keys = Nk;
    }
    if (B == 0) return 0;
    run_threads(fwd_worker, &J, n_threads);
    return J.status;
}

/* ------------------------------------------------------------------ decode */

typedef struct {
    const uint16_t *q, *kc, *vc;
    const int32_t *page_table, *seqlens;
    int page_size, B, Hq, Hkv, d, max_pages;
    double scale;
    double *o, *lse;
    int64_t next;
    int status;
} dec_job_t;

static void* dec_worker(void* p) {
    dec_job_t* J = (dec_job_t*)p;
    const int d = J->d, Hkv = J->Hkv, G = J->Hq / J->Hkv;
    for (;;) {
        const int64_t b = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (b >= J->B) break;
        const int64_t L = J->seqlens[b];
        if (L < 0 || L > (int64_t)J->max_pages * J->page_size) {
            __atomic_store_n(&J->status, -3, __ATOMIC_RELAXED);
            continue;
        }
        /* gather this sequence's cached rows, [L, Hkv, d], through the page table */
        const size_t row_elems = (size_t)Hkv * d;
        uint16_t* kb = (uint16_t*)malloc(sizeof(uint16_t) * row_elems * (size_t)(L > 0 ? L : 1));
        uint16_t* vb = (uint16_t*)malloc(sizeof(uint16_t) * row_elems * (size_t)(L > 0 ? L : 1));
        double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        if (!kb || !vb || !s || !qd) {
            __atomic_store_n(&J->status, -2, __ATOMIC_RELAXED);
            free(kb); free(vb); free(s); free(qd);
            continue;
        }
        for (int64_t t = 0; t < L; ++t) {
            const int64_t page = J->page_table[b * J->max_pages + t / J->page_size];
            const int64_t slot = t % J->page_size;
            const size_t src = (size_t)(page * J->page_size + slot) * row_elems;
            memcpy(kb + (size_t)t * row_elems, J->kc + src, sizeof(uint16_t) * row_elems);
            memcpy(vb + (size_t)t * row_elems, J->vc + src, sizeof(uint16_t) * row_elems);
        }
        for (int h = 0; h < J->Hq; ++h) {
            const int g = h / G;
            attend_row(J->q + (b * J->Hq + h) * d, kb + (size_t)g * d, vb + (size_t)g * d, (int64_t)row_elems, L, d,
                       J->scale, s, qd, J->o + (b * J->Hq + h) * d, J->lse + b * J->Hq + h);
        }
        free(kb); free(vb); free(s); free(qd);
    }
    return NULL;
}

/*
 * Paged decode. q: [B, Hq, d]; k_cache, v_cache: [num_pages, page_size, Hkv, d];
 * page_table: int32 [B, max_pages]; seqlens: int32 [B]. o: [B, Hq, d], lse: [B, Hq].
 * One query per sequence; all seqlens[b] cached keys are visible.
 */
int oracle_attn_decode_paged(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* page_table, const int32_t* seqlens, int page_size,
                             double* o, double* lse, int B, int Hq, int Hkv, int d, int max_pages,
                             double scale, int n_threads) {
    if (!q || !k_cache || !v_cache || !page_table || !seqlens || !o || !lse) return -1;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page_size <= 0 || max_pages < 0) return -1;
    dec_job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kc = k_cache; J.vc = v_cache; J.page_table = page_table; J.seqlens = seqlens;
    J.page_size = page_size; J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.d = d; J.max_pages = max_pages;
    J.scale = scale; J.o = o; J.lse = lse;
    if (B == 0) return 0;
    run_threads(dec_worker, &J, n_threads < B ? n_threads : B);
    return J.status;
}

/* ------------------------------------------------------------------ FP8 key/value caches */

/*
 * 8-bit floating-point caches ("Faster, more flexible FA4 for LLM inference", PR 2109:
 * inputs in 8-bit floating point with four or five exponent bits, e4m3 or e5m2). The
 * pages fix no scaling scheme; the reading taken is one descale factor per tensor: the
 * cached key with code c stands for k_descale * fp8(c), and likewise for values. fp8(c)
 * follows the OCP 8-bit floating-point definitions:
 *   fmt 0, e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
 *                subnormal, m/8 * 2^-6; S.1111.111 is NaN; no infinities (largest 448);
 *   fmt 1, e5m2: sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent 0 is
 *                subnormal, m/4 * 2^-14; exponent 31 is infinity (m = 0) or NaN.
 * The attention is the same three-pass definition, on these values in float64.
 */
double oracle_fp8_value(uint8_t c, int fmt) {
    const int neg = c >> 7;
    double v;
    if (fmt == 0) {
        const int e = (c >> 3) & 15, m = c & 7;
        if (e == 15 && m == 7) return NAN;
        v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    } else {
        const int e = (c >> 2) & 31, m = c & 3;
        if (e == 31) return m == 0 ? (neg ? -INFINITY : INFINITY) : NAN;
        v = e == 0 ? ldexp(m / 4.0, -14) : ldexp(1.0 + m / 4.0, e - 15);
    }
    return neg ? -v : v;
}

void oracle_fp8_values(const uint8_t* c, double* out, int64_t n, int fmt) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_value(c[i], fmt);
}

/* One query row (float64, d wide) against n keys (d wide, row stride kstride) and values
 * (dv wide, row stride vstride) given as float64 rows; o is dv wide. */
static void attend_row_f64(const double* qd, const double* k, const double* v, int64_t kstride, int64_t vstride,
                           int64_t n, int d, int dv, double scale, double* s, double* o, double* lse) {
    if (n <= 0) {
        for (int c = 0; c < dv; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qd[c] * k[j * kstride + c];
        s[j] = scale * acc;
    }
    double m = s[0];
    for (int64_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int c = 0; c < dv; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double p = exp(s[j] - m) / l;
        for (int c = 0; c < dv; ++c) o[c] += p * v[j * vstride + c];
    }
    *lse = m + log(l);
}

typedef struct {
    const uint16_t* q;
    const uint8_t *kc, *vc;
    int fmt;
    double k_descale, v_descale;
    const int32_t *page_table, *seqlens;
    int page_size, B, Hq, Hkv, d, max_pages;
    double scale;
    double *o, *lse;
    int64_t next;
    int status;
} dec8_job_t;

static void* dec8_worker(void* p) {
    dec8_job_t* J = (dec8_job_t*)p;
    const int d = J->d, Hkv = J->Hkv, G = J->Hq / J->Hkv;
    double ktab[256], vtab[256]; /* descale * fp8(c) for every code c */
    for (int c = 0; c < 256; ++c) {
        ktab[c] = J->k_descale * oracle_fp8_value((uint8_t)c, J->fmt);
        vtab[c] = J->v_descale * oracle_fp8_value((uint8_t)c, J->fmt);
    }
    for (;;) {
        const int64_t b = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (b >= J->B) break;
        const int64_t L = J->seqlens[b];
        if (L < 0 || L > (int64_t)J->max_pages * J->page_size) {
            __atomic_store_n(&J->status, -3, __ATOMIC_RELAXED);
            continue;
        }
        /* gather and widen this sequence's cached rows, [L, Hkv, d] */
        const size_t row_elems = (size_t)Hkv * d, n = (size_t)(L > 0 ? L : 1) * row_elems;
        double* kb = (double*)malloc(sizeof(double) * n);
        double* vb = (double*)malloc(sizeof(double) * n);
        double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        if (!kb || !vb || !s || !qd) {
            __atomic_store_n(&J->status, -2, __ATOMIC_RELAXED);
            free(kb); free(vb); free(s); free(qd);
            continue;
        }
        for (int64_t t = 0; t < L; ++t) {
            const int64_t page = J->page_table[b * J->max_pages + t / J->page_size];
            const size_t src = (size_t)(page * J->page_size + t % J->page_size) * row_elems;
            for (size_t e = 0; e < row_elems; ++e) {
                kb[(size_t)t * row_elems + e] = ktab[J->kc[src + e]];
                vb[(size_t)t * row_elems + e] = vtab[J->vc[src + e]];
            }
        }
        for (int h = 0; h < J->Hq; ++h) {
            const int g = h / G;
            for (int c = 0; c < d; ++c) qd[c] = bf16d(J->q[(b * J->Hq + h) * d + c]);
            attend_row_f64(qd, kb + (size_t)g * d, vb + (size_t)g * d, (int64_t)row_elems, (int64_t)row_elems, L, d, d,
                           J->scale, s, J->o + (b * J->Hq + h) * d, J->lse + b * J->Hq + h);
        }
        free(kb); free(vb); free(s); free(qd);
    }
    return NULL;
}

/*
 * Paged decode over FP8 caches. q: bf16 [B, Hq, d]; k_cache, v_cache: FP8 codes
 * [num_pages, page_size, Hkv, d]; fmt 0 = e4m3, 1 = e5m2; the rest as for
 * oracle_attn_decode_paged.
 */
int oracle_attn_decode_paged_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache, int fmt,
                                 double k_descale, double v_descale, const int32_t* page_table,
                                 const int32_t* seqlens, int page_size, double* o, double* lse, int B, int Hq,
                                 int Hkv, int d, int max_pages, double scale, int n_threads) {
    if (!q || !k_cache || !v_cache || !page_table || !seqlens || !o || !lse) return -1;
    if (fmt != 0 && fmt != 1) return -1;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page_size <= 0 || max_pages < 0) return -1;
    dec8_job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kc = k_cache; J.vc = v_cache; J.fmt = fmt; J.k_descale = k_descale; J.v_descale = v_descale;
    J.page_table = page_table; J.seqlens = seqlens; J.page_size = page_size; J.B = B; J.Hq = Hq; J.Hkv = Hkv;
    J.d = d; J.max_pages = max_pages; J.scale = scale; J.o = o; J.lse = lse;
    if (B == 0) return 0;
    run_threads(dec8_worker, &J, n_threads < B ? n_threads : B);
    return J.status;
}


/* ------------------------------------------------------------------ forward, float64 inputs */

/*
 * The forward definition on float64 inputs, for inputs that are not bf16: 8-bit
 * floating-point Q/K/V ("Faster, more flexible FA4 for LLM inference", PR 2109) are
 * decoded and multiplied by their descales by the caller, then passed here. Same
 * layouts, masks and rows as oracle_attn_fwd, except that values (and so outputs) may be
 * dv wide while queries and keys are d wide: head dims (d, dv) such as DeepSeek-V3's
 * (192, 128) ("FlashAttention-4: Blackwell algorithm-pipeline co-design", performance
 * section). The definition is unchanged: scores use d, the weighted sum runs over dv.
 */
static void* fwd_f64_worker(void* p) {
    fwd_job_t* J = (fwd_job_t*)p;
    const int d = J->d;
    const int G = J->Hq / J->Hkv;
    const int64_t total_tokens = J->cu ? J->cu[J->B] : (int64_t)J->B * J->Nq;
    const int64_t n_items = J->rows ? J->n_rows : total_tokens * J->Hq;
    double* s = (double*)malloc(sizeof(double) * (size_t)(J->max_keys > 0 ? J->max_keys : 1));
    if (!s) {
        __atomic_store_n(&J->status, -2, __ATOMIC_RELAXED);
        return NULL;
    }
    for (;;) {
        const int64_t it = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (it >= n_items) break;
        const int64_t row = J->rows ? J->rows[it] : it;
        const int64_t t = row / J->Hq;
        const int h = (int)(row % J->Hq);
        int64_t i, nq, nk, k0;
        if (row < 0 || locate(J, t, &i, &nq, &nk, &k0) != 0) {
            __atomic_store_n(&J->status, -3, __ATOMIC_RELAXED);
            continue;
        }
        int64_t n_vis = nk;
        if (J->causal) {
            const int64_t last = i + (nk - nq);
            n_vis = last + 1 < nk ? last + 1 : nk;
        }
        if (n_vis < 0) n_vis = 0;
        const int g = h / G;
        const int dv = J->dv;
        const int64_t k_stride = (int64_t)J->Hkv * d, v_stride = (int64_t)J->Hkv * dv;
        attend_row_f64(J->qf + (t * J->Hq + h) * d, J->kf + k0 * k_stride + (int64_t)g * d,
                       J->vf + k0 * v_stride + (int64_t)g * dv, k_stride, v_stride, n_vis, d, dv, J->scale, s,
                       J->o + it * dv, J->lse + it);
    }
    free(s);
    return NULL;
}

int oracle_attn_fwd_f64(const double* q, const double* k, const double* v, double* o, double* lse, int B, int Hq,
                        int Hkv, int Nq, int Nk, int d, int dv, double scale, int causal, const int32_t* cu_seqlens,
                        const int64_t* rows, int64_t n_rows, int n_threads) {
    if (!q || !k || !v || !o || !lse || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || dv <= 0) return -1;
    fwd_job_t J;
    memset(&J, 0, sizeof J);
    J.qf = q; J.kf = k; J.vf = v; J.o = o; J.lse = lse;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.Nq = Nq; J.Nk = Nk; J.d = d; J.dv = dv; J.causal = causal;
    J.scale = scale; J.cu = cu_seqlens; J.rows = rows; J.n_rows = n_rows;
    if (cu_seqlens) {
        int64_t mx = 0;
        for (int b = 0; b < B; ++b) {
            const int64_t L = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
            if (L < 0) return -1;
            if (L > mx) mx = L;
        }
        J.max_keys = mx;
    } else {
        if (Nq < 0 || Nk < 0) return -1;
        J.max_keys = Nk;
    }
    if (B == 0) return 0;
    run_threads(fwd_f64_worker, &J, n_threads);
    return J.status;
}
