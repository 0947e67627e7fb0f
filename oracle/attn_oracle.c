/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, no fusion):
 *   "FlashAttention 1-4 详解" (pinghaoyang.com.cn), section 原算法 -- the standard
 *   attention S = Q K^T, P = softmax(S / sqrt(d)), O = P V, written there as one
 *   formula and as the three-step S/P/O pipeline.  The scale is an argument
 *   (default 1/sqrt(d)) and is applied to the scores before the softmax.
 *   The softmax of one row is the numerically stable two-pass form of the same
 *   page's "Online Softmax 数学推导" section: m = max_k x_k, then
 *   e^{x_i - m} / sum_j e^{x_j - m}.
 *   The per-row log-sum-exp that the fused kernel outputs (the softmax_lse kept
 *   for the backward pass, "flash-attention" (ai-reference-codex.pages.dev),
 *   sections 2.1 and 2.3) is LSE = m + ln(sum_j e^{x_j - m}), natural log of the
 *   sum of exponentials of the scaled scores.
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *   - causal masking is aligned bottom-right: query i of Nq may see key j of Nk when
 *     j <= i + (Nk - Nq); for Nq == Nk this is j <= i ("FlashAttention 1-4 详解",
 *     FlashAttention 2 engineering notes, causal lower triangle);
 *   - a row with no visible key has O = 0 and LSE = -inf;
 *   - grouped-query attention maps query head h to key/value head h / (Hq / Hkv)
 *     ("flash-attention", capabilities table, MQA / GQA row: Hkv divides Hq);
 *   - variable-length batches are packed along the token axis and delimited by the
 *     prefix sums cu_seqlens ("flash-attention", capabilities table, varlen row);
 *   - single-query decode attends to the first cache_seqlens[b] rows of the cache
 *     ("flash-attention", capabilities table, KV cache row; section 1 usage); the query
 *     sits at position cache_seqlens[b] - 1 (bottom-right alignment with Nq = 1).
 *
 * Score modifiers ("flash-attention", capabilities table: causal / sliding window /
 * ALiBi / softcap; the pages name them and give no formulas, so the plain readings
 * below are taken).  With pos = i + (Nk - Nq) the bottom-right position of query i:
 *   - sliding window (wl, wr): key j is visible when pos - wl <= j <= pos + wr; a
 *     negative bound is unbounded; causal is the window (-1, 0);
 *   - softcap c > 0: the scaled score z = scale * q . k_j becomes c * tanh(z / c);
 *   - ALiBi slope a (per batch and query head): the score (after the softcap) gets
 *     - a * |pos - j| added.
 * The softmax and the log-sum-exp are then taken over the modified scores of the
 * visible keys.
 *
 * Inputs are 16-bit float bit patterns (uint16): bf16 (elem = 0) or IEEE binary16
 * (elem = 1), the two element types of the fused kernels ("flash-attention", section 5:
 * fp16 / bf16 only).  Each is widened exactly to double, so the oracle sees the same
 * numbers the GPU sees; all arithmetic is IEEE double.
 * Work is spread over threads by query row; the arithmetic of a row does not depend
 * on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bits -> exact double (bf16 is the upper half of an IEEE binary32). */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 bits -> exact double: sign, 5-bit exponent (bias 15), 10-bit fraction. */
static double fp16_to_double(uint16_t bits) {
    int sign = bits >> 15, e = (bits >> 10) & 0x1f, f = bits & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(f | 0x400), e - 25);           /* (1024 + f) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

/* Element type of the current job (0 bf16, 1 fp16); set per call before any worker runs. */
static double widen(uint16_t bits, int elem) {
    return elem ? fp16_to_double(bits) : bf16_to_double(bits);
}

/* Score modifiers of one row: softcap (0 = off) and the ALiBi slope (has_alibi). */
typedef struct {
    double softcap;
    int has_alibi;
    double slope;
} score_mod_t;

/*
 * One query row against the visible keys lo..hi-1.
 * q      : d values
 * krow(j): key j at kbase + j * k_stride, d values
 * vrow(j): value j at vbase + j * v_stride, d values
 * pos    : bottom-right position of the query (for the ALiBi distance)
 * s      : scratch of hi - lo doubles; on return it holds the probabilities P_j
 * o      : d doubles, o = sum_j P_j v_j
 * lse    : natural-log sum of exp of the (modified) scaled scores
 */
static void attend_row(const uint16_t *q, const uint16_t *kbase, int64_t k_stride,
                       const uint16_t *vbase, int64_t v_stride, int64_t lo, int64_t hi,
                       int64_t pos, int d, double scale, const score_mod_t *mod, int elem,
                       double *s, double *o, double *lse) {
    int64_t nkeys = hi - lo;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (nkeys <= 0) {
        *lse = -INFINITY;
        return;
    }
    /* S = scale * q . k_j, then the softcap and the ALiBi bias */
    for (int64_t j = lo; j < hi; ++j) {
        const uint16_t *kr = kbase + j * k_stride;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += widen(q[c], elem) * widen(kr[c], elem);
        double z = scale * acc;
        if (mod->softcap > 0.0) z = mod->softcap * tanh(z / mod->softcap);
        if (mod->has_alibi) z -= mod->slope * fabs((double)(pos - j));
        s[j - lo] = z;
    }
    /* stable softmax: m = max_j s_j, l = sum_j e^{s_j - m}, P_j = e^{s_j - m} / l */
    double m = s[0];
    for (int64_t j = 1; j < nkeys; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < nkeys; ++j) s[j] /= l;
    /* O = P V */
    for (int64_t j = 0; j < nkeys; ++j) {
        const uint16_t *vr = vbase + (lo + j) * v_stride;
        for (int c = 0; c < d; ++c) o[c] += s[j] * widen(vr[c], elem);
    }
    *lse = m + log(l);
}

/*
 * Keys visible to the query at bottom-right position pos among Nk keys under the window
 * (wl, wr) (negative = unbounded): [*lo, *hi), empty when *hi <= *lo.
 */
static void visible_range(int64_t pos, int64_t Nk, int64_t wl, int64_t wr, int64_t *lo,
                          int64_t *hi) {
    int64_t a = 0, b = Nk;
    if (wl >= 0 && pos - wl > a) a = pos - wl;
    if (wr >= 0 && pos + wr + 1 < b) b = pos + wr + 1;
    *lo = a;
    *hi = b > a ? b : a;
}

/* ------------------------------------------------------------------------- */
/* Work description shared by the threaded drivers.                          */

typedef struct {
    /* dense layout: element (b, n, h, c) at base + b*s[0] + n*s[1] + h*s[2] + c */
    const uint16_t *q, *k, *v;
    int64_t qs[3], ks[3], vs[3];
    int B, Nq, Nk, Hq, Hkv, d;
    double scale;
    /* window bounds (causal already folded in as wr = 0), softcap, ALiBi slopes
       (slope of (b, h) at alibi[b * alibi_sb + h], NULL = none) */
    int64_t wl, wr;
    double softcap;
    const double *alibi;
    int64_t alibi_sb;
    /* varlen: prefix sums over the packed token axis (B+1 entries) */
    const int32_t *cu_q, *cu_k;
    /* kv cache: visible prefix length per batch entry */
    const int32_t *cache_len;
    /* optional list of (b, h, i) triples; when set only those rows are computed */
    const int32_t *rows;
    int64_t nrows;
    /* outputs */
    double *o, *lse;
    int64_t os[3];      /* output strides (b, n, h) for the full drivers */
    int64_t lse_s[3];   /* lse strides (b, h, n) */
    int mode;           /* 0 dense, 1 varlen, 2 kvcache */
    int elem;           /* 0 bf16, 1 fp16 */
    int nthreads, tid;
    int64_t total;      /* number of (b, h, i) work items */
} job_t;

/* Map a flat work index to (b, h, i) for the full drivers. */
static void decode_index(const job_t *J, int64_t w, int *b, int *h, int64_t *i) {
    if (J->rows) {
        *b = J->rows[3 * w];
        *h = J->rows[3 * w + 1];
        *i = J->rows[3 * w + 2];
        return;
    }
    if (J->mode == 1) {
        /* varlen: w runs over (token t of the packed batch, head h) */
        int64_t t = w / J->Hq;
        *h = (int)(w % J->Hq);
        int bb = 0;
        while (J->cu_q[bb + 1] <= t) ++bb;
        *b = bb;
        *i = t - J->cu_q[bb];
        return;
    }
    int64_t per_b = (int64_t)J->Nq * J->Hq;
    *b = (int)(w / per_b);
    int64_t r = w % per_b;
    *i = r / J->Hq;
    *h = (int)(r % J->Hq);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    int64_t max_keys = J->Nk;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    double *orow = (double *)malloc(sizeof(double) * (size_t)J->d);
    int group = J->Hq / J->Hkv;
    for (int64_t w = J->tid; w < J->total; w += J->nthreads) {
        int b, h;
        int64_t i;
        decode_index(J, w, &b, &h, &i);
        int g = h / group; /* key/value head shared by this query head */
        const uint16_t *qrow, *kbase, *vbase;
        int64_t nk, pos, k_stride, v_stride;
        if (J->mode == 0) {
            qrow = J->q + b * J->qs[0] + i * J->qs[1] + h * J->qs[2];
            kbase = J->k + b * J->ks[0] + g * J->ks[2];
            vbase = J->v + b * J->vs[0] + g * J->vs[2];
            k_stride = J->ks[1];
            v_stride = J->vs[1];
            pos = i + (J->Nk - J->Nq);
            nk = J->Nk;
        } else if (J->mode == 1) {
            int64_t nq = J->cu_q[b + 1] - J->cu_q[b];
            nk = J->cu_k[b + 1] - J->cu_k[b];
            qrow = J->q + (J->cu_q[b] + i) * J->qs[1] + h * J->qs[2];
            kbase = J->k + J->cu_k[b] * J->ks[1] + g * J->ks[2];
            vbase = J->v + J->cu_k[b] * J->vs[1] + g * J->vs[2];
            k_stride = J->ks[1];
            v_stride = J->vs[1];
            pos = i + (nk - nq);
        } else {
            /* decode: one query per batch entry, the last of a sequence of cache_len[b] */
            qrow = J->q + b * J->qs[0] + h * J->qs[2];
            kbase = J->k + b * J->ks[0] + g * J->ks[2];
            vbase = J->v + b * J->vs[0] + g * J->vs[2];
            k_stride = J->ks[1];
            v_stride = J->vs[1];
            nk = J->cache_len[b];
            pos = nk - 1;
        }
        int64_t lo, hi;
        visible_range(pos, nk, J->wl, J->wr, &lo, &hi);
        score_mod_t mod;
        mod.softcap = J->softcap;
        mod.has_alibi = J->alibi != NULL;
        mod.slope = J->alibi ? J->alibi[b * J->alibi_sb + h] : 0.0;
        double lse;
        attend_row(qrow, kbase, k_stride, vbase, v_stride, lo, hi, pos, J->d, J->scale, &mod,
                   J->elem, s, orow, &lse);
        double *odst;
        double *ldst;
        if (J->rows) {
            odst = J->o + w * J->d;
            ldst = J->lse + w;
        } else if (J->mode == 1) {
            int64_t t = J->cu_q[b] + i;
            odst = J->o + t * J->os[1] + h * J->os[2];
            ldst = J->lse + h * J->lse_s[1] + t * J->lse_s[2];
        } else {
            odst = J->o + b * J->os[0] + i * J->os[1] + h * J->os[2];
            ldst = J->lse + b * J->lse_s[0] + h * J->lse_s[1] + i * J->lse_s[2];
        }
        memcpy(odst, orow, sizeof(double) * (size_t)J->d);
        *ldst = lse;
    }
    free(s);
    free(orow);
    return NULL;
}

static int run_threads(job_t *base) {
    int n = base->nthreads < 1 ? 1 : base->nthreads;
    if (n > 512) n = 512;
    pthread_t th[512];
    job_t jobs[512];
    for (int t = 0; t < n; ++t) {
        jobs[t] = *base;
        jobs[t].nthreads = n;
        jobs[t].tid = t;
    }
    for (int t = 1; t < n; ++t)
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) return -1;
    worker(&jobs[0]);
    for (int t = 1; t < n; ++t) pthread_join(th[t], NULL);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Exported entry points (called through ctypes by oracle/oracle.py).        */
/*
 * Every entry point ends with the element type and the score modifiers:
 *   elem          : 0 bf16, 1 fp16
 *   window_left/right : sliding-window bounds, negative = unbounded (causal != 0 sets the
 *                   right bound to 0)
 *   softcap       : 0 = off, else > 0
 *   alibi         : NULL or per-(batch, query head) slopes, slope of (b, h) at
 *                   alibi[b * alibi_sb + h] (alibi_sb = 0 shares one row of Hq slopes)
 */

static int set_common(job_t *J, int Hq, int Hkv, int d, int elem, int causal, int window_left,
                      int window_right, double softcap, const double *alibi, int64_t alibi_sb) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || elem < 0 || elem > 1) return -1;
    if (!(softcap >= 0.0) || alibi_sb < 0) return -1;
    J->elem = elem;
    J->wl = window_left < 0 ? -1 : window_left;
    J->wr = causal ? 0 : (window_right < 0 ? -1 : window_right);
    J->softcap = softcap;
    J->alibi = alibi;
    J->alibi_sb = alibi_sb;
    return 0;
}

/*
 * Dense batched attention.  q: [B, Nq, Hq, d], k/v: [B, Nk, Hkv, d] with element
 * strides (b, n, h) given, unit stride over d.  o: [B, Nq, Hq, d] contiguous
 * doubles, lse: [B, Hq, Nq] contiguous doubles.  Returns 0 on success.
 */
int oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Nq, int Nk,
               int Hq, int Hkv, int d, const int64_t *q_strides, const int64_t *k_strides,
               const int64_t *v_strides, double scale, int causal, double *o, double *lse,
               int nthreads, int elem, int window_left, int window_right, double softcap,
               const double *alibi, int64_t alibi_sb) {
    job_t J;
    memset(&J, 0, sizeof J);
    if (set_common(&J, Hq, Hkv, d, elem, causal, window_left, window_right, softcap, alibi,
                   alibi_sb) != 0)
        return -1;
    J.q = q; J.k = k; J.v = v;
    for (int a = 0; a < 3; ++a) { J.qs[a] = q_strides[a]; J.ks[a] = k_strides[a]; J.vs[a] = v_strides[a]; }
    J.B = B; J.Nq = Nq; J.Nk = Nk; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.scale = scale;
    J.o = o; J.lse = lse;
    J.os[0] = (int64_t)Nq * Hq * d; J.os[1] = (int64_t)Hq * d; J.os[2] = d;
    J.lse_s[0] = (int64_t)Hq * Nq; J.lse_s[1] = Nq; J.lse_s[2] = 1;
    J.mode = 0;
    J.nthreads = nthreads;
    J.total = (int64_t)B * Nq * Hq;
    return run_threads(&J);
}

/*
 * Dense attention on a chosen set of rows: rows is n triples (b, h, i).
 * o: [n, d] doubles, lse: [n] doubles.
 */
int oracle_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Nq, int Nk,
                    int Hq, int Hkv, int d, const int64_t *q_strides, const int64_t *k_strides,
                    const int64_t *v_strides, double scale, int causal, const int32_t *rows,
                    int64_t n, double *o, double *lse, int nthreads, int elem, int window_left,
                    int window_right, double softcap, const double *alibi, int64_t alibi_sb) {
    job_t J;
    memset(&J, 0, sizeof J);
    if (set_common(&J, Hq, Hkv, d, elem, causal, window_left, window_right, softcap, alibi,
                   alibi_sb) != 0)
        return -1;
    J.q = q; J.k = k; J.v = v;
    for (int a = 0; a < 3; ++a) { J.qs[a] = q_strides[a]; J.ks[a] = k_strides[a]; J.vs[a] = v_strides[a]; }
    J.B = B; J.Nq = Nq; J.Nk = Nk; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.scale = scale;
    J.rows = rows; J.nrows = n;
    J.o = o; J.lse = lse;
    J.mode = 0;
    J.nthreads = nthreads;
    J.total = n;
    return run_threads(&J);
}

/*
 * Packed variable-length batch.  q: [total_q, Hq, d], k/v: [total_k, Hkv, d] with
 * token and head strides given ((b) stride unused); cu_q, cu_k: B+1 prefix sums
 * (host memory).  o: [total_q, Hq, d] doubles, lse: [Hq, total_q] doubles.
 */
int oracle_fwd_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *cu_q, const int32_t *cu_k, int B, int Hq, int Hkv, int d,
                      const int64_t *q_strides, const int64_t *k_strides, const int64_t *v_strides,
                      double scale, int causal, double *o, double *lse, int nthreads, int elem,
                      int window_left, int window_right, double softcap, const double *alibi,
                      int64_t alibi_sb) {
    job_t J;
    memset(&J, 0, sizeof J);
    if (set_common(&J, Hq, Hkv, d, elem, causal, window_left, window_right, softcap, alibi,
                   alibi_sb) != 0)
        return -1;
    J.q = q; J.k = k; J.v = v;
    for (int a = 0; a < 3; ++a) { J.qs[a] = q_strides[a]; J.ks[a] = k_strides[a]; J.vs[a] = v_strides[a]; }
    int64_t total_q = cu_q[B];
    int max_k = 0;
    for (int b = 0; b < B; ++b) {
        int nk = cu_k[b + 1] - cu_k[b];
        if (nk > max_k) max_k = nk;
    }
    J.B = B; J.Nq = 0; J.Nk = max_k; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.scale = scale;
    J.cu_q = cu_q; J.cu_k = cu_k;
    J.o = o; J.lse = lse;
    J.os[0] = 0; J.os[1] = (int64_t)Hq * d; J.os[2] = d;
    J.lse_s[0] = 0; J.lse_s[1] = total_q; J.lse_s[2] = 1;
    J.mode = 1;
    J.nthreads = nthreads;
    J.total = total_q * Hq;
    return run_threads(&J);
}

/*
 * Single-query decode over a padded KV cache.  q: [B, 1, Hq, d] (strides given),
 * k/v cache: [B, Lmax, Hkv, d] (strides given), cache_len: B visible lengths.
 * o: [B, Hq, d] doubles, lse: [B, Hq] doubles.  The query is the last token of its
 * sequence, so only the left window bound can hide a cached key.
 */
int oracle_fwd_kvcache(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                       const int32_t *cache_len, int B, int Lmax, int Hq, int Hkv, int d,
                       const int64_t *q_strides, const int64_t *k_strides, const int64_t *v_strides,
                       double scale, double *o, double *lse, int nthreads, int elem,
                       int window_left, int window_right, double softcap, const double *alibi,
                       int64_t alibi_sb) {
    job_t J;
    memset(&J, 0, sizeof J);
    if (set_common(&J, Hq, Hkv, d, elem, 0, window_left, window_right, softcap, alibi,
                   alibi_sb) != 0)
        return -1;
    for (int b = 0; b < B; ++b)
        if (cache_len[b] < 0 || cache_len[b] > Lmax) return -1;
    J.q = q; J.k = kc; J.v = vc;
    for (int a = 0; a < 3; ++a) { J.qs[a] = q_strides[a]; J.ks[a] = k_strides[a]; J.vs[a] = v_strides[a]; }
    J.B = B; J.Nq = 1; J.Nk = Lmax; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.scale = scale;
    J.cache_len = cache_len;
    J.o = o; J.lse = lse;
    J.os[0] = (int64_t)Hq * d; J.os[1] = 0; J.os[2] = d;
    J.lse_s[0] = Hq; J.lse_s[1] = 1; J.lse_s[2] = 0;
    J.mode = 2;
    J.nthreads = nthreads;
    J.total = (int64_t)B * Hq;
    return run_threads(&J);
}

/*
 * Probabilities of one dense row (b, h, i): P_j for j < Nk (0 for keys the row may
 * not see).  Exposed so that tests can check invariants of P itself on tiny cases.
 */
int oracle_row_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Nq, int Nk,
                     int Hq, int Hkv, int d, const int64_t *q_strides, const int64_t *k_strides,
                     const int64_t *v_strides, double scale, int causal, int b, int h, int i,
                     double *p_out, int elem, int window_left, int window_right, double softcap,
                     const double *alibi, int64_t alibi_sb) {
    job_t J;
    memset(&J, 0, sizeof J);
    if (set_common(&J, Hq, Hkv, d, elem, causal, window_left, window_right, softcap, alibi,
                   alibi_sb) != 0)
        return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Nq) return -1;
    int g = h / (Hq / Hkv);
    int64_t pos = (int64_t)i + (Nk - Nq), lo, hi;
    visible_range(pos, Nk, J.wl, J.wr, &lo, &hi);
    score_mod_t mod;
    mod.softcap = softcap;
    mod.has_alibi = alibi != NULL;
    mod.slope = alibi ? alibi[b * alibi_sb + h] : 0.0;
    double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
    double lse;
    attend_row(q + b * q_strides[0] + (int64_t)i * q_strides[1] + h * q_strides[2],
               k + b * k_strides[0] + g * k_strides[2], k_strides[1],
               v + b * v_strides[0] + g * v_strides[2], v_strides[1], lo, hi, pos, d, scale,
               &mod, elem, s, orow, &lse);
    for (int64_t j = 0; j < Nk; ++j) p_out[j] = (j >= lo && j < hi) ? s[j - lo] : 0.0;
    free(s);
    free(orow);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* KV-cache extras: rotary embedding of the new key and the query.            */
/*
 * "flash-attention" (section 1, usage: the decode call updates the KV cache in place and
 * applies rotary in the same step; capabilities table, KV cache row).  The pages give no
 * formula; the rotation read here is the standard rotary position embedding: dimension
 * pairs (a, b) of the first rotary_dim dimensions -- (i, i + rotary_dim/2), or (2i, 2i+1)
 * when interleaved -- turn by the angle whose cosine and sine are the table entries of
 * the token's position p:
 *     y_a = x_a cos - x_b sin,   y_b = x_a sin + x_b cos.
 * Dimensions from rotary_dim on are copied.  The result is stored in the element type of
 * the cache, so it is rounded once, to nearest even.  Because that rounding turns a real
 * number into a 16-bit code, it is evaluated in the precision the kernel uses: fp32, with
 * the products and sums grouped as written below (one fused multiply-add per output), so
 * that both sides round the same fp32 value.
 */

/* fp32 -> bf16 bits, round to nearest even (NaN stays NaN). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* fp32 -> IEEE binary16 bits, round to nearest even, with subnormals and overflow to inf. */
static uint16_t f32_to_fp16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);          /* NaN */
    if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);         /* rounds to >= 65520: inf */
    int e = (int)(a >> 23) - 127;                                    /* unbiased exponent */
    uint32_t m = (a & 0x7fffffu) | 0x800000u;                        /* 24-bit significand */
    if (a < 0x00800000u) return sign;                                /* fp32 subnormal: far below fp16 */
    int shift;                                                       /* bits to drop */
    uint32_t base;
    if (e >= -14) {                                                  /* fp16 normal */
        shift = 13;
        base = (uint32_t)(e + 15) << 10;
        m &= 0x7fffffu;                                              /* drop the implicit one */
    } else {                                                         /* fp16 subnormal: units of 2^-24 */
        shift = 13 + (-14 - e);
        if (shift > 24) return sign;
        base = 0;
    }
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | (base + q));                            /* a carry moves into the exponent */
}

static uint16_t f32_to_bits(float f, int elem) {
    return elem ? f32_to_fp16_bits(f) : f32_to_bf16_bits(f);
}

/*
 * Rotary embedding of `rows` vectors of d elements: row r at x + r * x_stride, position
 * pos[r], tables cos/sin [*, rotary_dim / 2] fp32 (row p at p * rotary_dim / 2).  Writes
 * out (row r at out + r * d, contiguous).  Returns 0, or -1 on bad arguments.
 */
int oracle_rotary(const uint16_t *x, int64_t x_stride, int64_t rows, int d, const int32_t *pos,
                  const float *cos_t, const float *sin_t, int rotary_dim, int interleaved,
                  uint16_t *out, int elem) {
    if (d <= 0 || rotary_dim <= 0 || rotary_dim > d || (rotary_dim & 1) || elem < 0 || elem > 1)
        return -1;
    int half = rotary_dim / 2;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * x_stride;
        uint16_t *orow = out + r * d;
        for (int c = 0; c < d; ++c) orow[c] = xr[c];
        const float *cr = cos_t + (int64_t)pos[r] * half;
        const float *sr = sin_t + (int64_t)pos[r] * half;
        for (int i = 0; i < half; ++i) {
            int ia = interleaved ? 2 * i : i;
            int ib = interleaved ? 2 * i + 1 : i + half;
            float xa = (float)widen(xr[ia], elem), xb = (float)widen(xr[ib], elem);
            float c = cr[i], s = sr[i];
            float ya = fmaf(xa, c, -(xb * s));
            float yb = fmaf(xa, s, xb * c);
            orow[ia] = f32_to_bits(ya, elem);
            orow[ib] = f32_to_bits(yb, elem);
        }
    }
    return 0;
}

/* fp32 values -> 16-bit codes (round to nearest even), exposed for the pins. */
int oracle_round16(const float *x, int64_t n, uint16_t *out, int elem) {
    if (elem < 0 || elem > 1) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bits(x[i], elem);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward pass.                                                             */
/*
 * Gradients of the attention output with respect to Q, K and V for an upstream gradient
 * dO ("flash-attention", sections 2.3 and 4: the backward pass keeps only q, k, v, out
 * and softmax_lse and recomputes P = exp(S * scale - LSE); "FlashAttention 1-4 详解",
 * FlashAttention 2: parallel over K/V column blocks, dK and dV accumulated per key,
 * dQ accumulated across key blocks).  The plain chain rule through O = P V,
 * P = softmax(S), S = scale Q K^T:
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . v_j
 *     D_i   = sum_j P_ij dP_ij          (= dO_i . O_i)
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j  = scale sum_i dS_ij q_i
 * Masked pairs have P = 0 and contribute nothing; with grouped-query attention dK and dV
 * of a key/value head sum over the query heads that read it.
 * With the score modifiers the softmax runs over z_ij (window, softcap, ALiBi as in the
 * forward) and the chain rule passes through z(s), s = scale q . k: the ALiBi bias does not
 * depend on q or k, a softcap c gives dz/ds = 1 - tanh^2(s / c), so dS above becomes
 * P_ij (dP_ij - D_i) dz/ds before it enters dQ and dK.
 * Two passes, each over independent items: pass 1 per query row (its LSE, D_i and
 * dQ_i), pass 2 per key row (dK_j and dV_j, with P recomputed from pass 1's LSE).
 */

typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int64_t qs[3], ks[3], vs[3], dos[3];
    int B, Nq, Nk, Hq, Hkv, d, elem;
    double scale;
    int64_t wl, wr;           /* window bounds (causal folded in as wr = 0), -1 = unbounded */
    double softcap;
    const double *alibi;      /* slope of (b, h) at alibi[b * alibi_sb + h], or NULL */
    int64_t alibi_sb;
    double *lse, *D;          /* [B, Hq, Nq] (pass 1 output, pass 2 input) */
    double *dq, *dk, *dv;     /* contiguous [B, N, H, d] */
    int pass, nthreads, tid;
} bwd_job_t;

static double dot16(const uint16_t *a, const uint16_t *b, int d, int elem) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += widen(a[c], elem) * widen(b[c], elem);
    return acc;
}

/* Modified score z of raw dot product acc for query position pos and key j, and dz/ds. */
static double bwd_score(const bwd_job_t *J, double acc, double slope, int64_t pos, int64_t j,
                        double *dzds) {
    double z = J->scale * acc;
    *dzds = 1.0;
    if (J->softcap > 0.0) {
        double t = tanh(z / J->softcap);
        z = J->softcap * t;
        *dzds = 1.0 - t * t;
    }
    if (J->alibi) z -= slope * fabs((double)(pos - j));
    return z;
}

static void *bwd_worker(void *arg) {
    bwd_job_t *J = (bwd_job_t *)arg;
    const int d = J->d, G = J->Hq / J->Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Nk > 0 ? J->Nk : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(J->Nk > 0 ? J->Nk : 1));
    if (J->pass == 1) {
        int64_t total = (int64_t)J->B * J->Hq * J->Nq;
        for (int64_t w = J->tid; w < total; w += J->nthreads) {
            int b = (int)(w / ((int64_t)J->Hq * J->Nq));
            int h = (int)((w / J->Nq) % J->Hq);
            int64_t i = w % J->Nq, g = h / G, pos = i + (J->Nk - J->Nq), lo, hi;
            visible_range(pos, J->Nk, J->wl, J->wr, &lo, &hi);
            int64_t n = hi - lo;
            double slope = J->alibi ? J->alibi[b * J->alibi_sb + h] : 0.0;
            const uint16_t *qi = J->q + b * J->qs[0] + i * J->qs[1] + h * J->qs[2];
            const uint16_t *doi = J->dout + b * J->dos[0] + i * J->dos[1] + h * J->dos[2];
            double *dqi = J->dq + (((int64_t)b * J->Nq + i) * J->Hq + h) * d;
            int64_t li = ((int64_t)b * J->Hq + h) * J->Nq + i;
            for (int c = 0; c < d; ++c) dqi[c] = 0.0;
            if (n == 0) { J->lse[li] = -INFINITY; J->D[li] = 0.0; continue; }
            double m = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                int64_t j = lo + t;
                double dz;
                s[t] = bwd_score(J, dot16(qi, J->k + b * J->ks[0] + j * J->ks[1] + g * J->ks[2], d,
                                          J->elem), slope, pos, j, &dz);
                if (s[t] > m) m = s[t];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double e = exp(s[j] - m);
                s[j] = e;
                l += e;
            }
            double Di = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                int64_t j = lo + t;
                s[t] /= l;                                                   /* P_ij */
                dp[t] = dot16(doi, J->v + b * J->vs[0] + j * J->vs[1] + g * J->vs[2], d, J->elem);
                Di += s[t] * dp[t];
            }
            for (int64_t t = 0; t < n; ++t) {
                int64_t j = lo + t;
                const uint16_t *kj = J->k + b * J->ks[0] + j * J->ks[1] + g * J->ks[2];
                double dz;
                bwd_score(J, dot16(qi, kj, d, J->elem), slope, pos, j, &dz);
                double ds = s[t] * (dp[t] - Di) * dz;
                for (int c = 0; c < d; ++c) dqi[c] += J->scale * ds * widen(kj[c], J->elem);
            }
            J->lse[li] = m + log(l);
            J->D[li] = Di;
        }
    } else {
        int64_t total = (int64_t)J->B * J->Hkv * J->Nk;
        for (int64_t w = J->tid; w < total; w += J->nthreads) {
            int b = (int)(w / ((int64_t)J->Hkv * J->Nk));
            int g = (int)((w / J->Nk) % J->Hkv);
            int64_t j = w % J->Nk;
            const uint16_t *kj = J->k + b * J->ks[0] + j * J->ks[1] + g * J->ks[2];
            const uint16_t *vj = J->v + b * J->vs[0] + j * J->vs[1] + g * J->vs[2];
            double *dkj = J->dk + (((int64_t)b * J->Nk + j) * J->Hkv + g) * d;
            double *dvj = J->dv + (((int64_t)b * J->Nk + j) * J->Hkv + g) * d;
            for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
            for (int h = g * G; h < (g + 1) * G; ++h) {
                double slope = J->alibi ? J->alibi[b * J->alibi_sb + h] : 0.0;
                for (int64_t i = 0; i < J->Nq; ++i) {
                    int64_t pos = i + (J->Nk - J->Nq), lo, hi;
                    visible_range(pos, J->Nk, J->wl, J->wr, &lo, &hi);
                    if (j < lo || j >= hi) continue;
                    int64_t li = ((int64_t)b * J->Hq + h) * J->Nq + i;
                    const uint16_t *qi = J->q + b * J->qs[0] + i * J->qs[1] + h * J->qs[2];
                    const uint16_t *doi = J->dout + b * J->dos[0] + i * J->dos[1] + h * J->dos[2];
                    double dz;
                    double z = bwd_score(J, dot16(qi, kj, d, J->elem), slope, pos, j, &dz);
                    double p = exp(z - J->lse[li]);
                    double ds = p * (dot16(doi, vj, d, J->elem) - J->D[li]) * dz;
                    for (int c = 0; c < d; ++c) {
                        dvj[c] += p * widen(doi[c], J->elem);
                        dkj[c] += J->scale * ds * widen(qi[c], J->elem);
                    }
                }
            }
        }
    }
    free(s);
    free(dp);
    return NULL;
}

static int bwd_run(bwd_job_t *base) {
    int n = base->nthreads < 1 ? 1 : (base->nthreads > 512 ? 512 : base->nthreads);
    pthread_t th[512];
    bwd_job_t jobs[512];
    for (int t = 0; t < n; ++t) { jobs[t] = *base; jobs[t].nthreads = n; jobs[t].tid = t; }
    for (int t = 1; t < n; ++t)
        if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) return -1;
    bwd_worker(&jobs[0]);
    for (int t = 1; t < n; ++t) pthread_join(th[t], NULL);
    return 0;
}

/*
 * Backward of dense batched attention.  q, dout: [B, Nq, Hq, d]; k, v: [B, Nk, Hkv, d]
 * (element strides (b, n, h) given).  Outputs, contiguous doubles: dq [B, Nq, Hq, d],
 * dk, dv [B, Nk, Hkv, d], and the lse and D = rowsum(dO * O) of each row [B, Hq, Nq].
 */
int oracle_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
               int B, int Nq, int Nk, int Hq, int Hkv, int d, const int64_t *q_strides,
               const int64_t *k_strides, const int64_t *v_strides, const int64_t *do_strides,
               double scale, int causal, double *dq, double *dk, double *dv, double *lse,
               double *D, int nthreads, int elem, int window_left, int window_right,
               double softcap, const double *alibi, int64_t alibi_sb) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || elem < 0 || elem > 1) return -1;
    if (!(softcap >= 0.0) || alibi_sb < 0) return -1;
    bwd_job_t J;
    memset(&J, 0, sizeof J);
    J.wl = window_left < 0 ? -1 : window_left;
    J.wr = causal ? 0 : (window_right < 0 ? -1 : window_right);
    J.softcap = softcap;
    J.alibi = alibi;
    J.alibi_sb = alibi_sb;
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    for (int a = 0; a < 3; ++a) {
        J.qs[a] = q_strides[a]; J.ks[a] = k_strides[a]; J.vs[a] = v_strides[a];
        J.dos[a] = do_strides[a];
    }
    J.B = B; J.Nq = Nq; J.Nk = Nk; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.elem = elem; J.scale = scale;
    J.lse = lse; J.D = D; J.dq = dq; J.dk = dk; J.dv = dv;
    J.nthreads = nthreads;
    J.pass = 1;
    if (bwd_run(&J) != 0) return -1;
    J.pass = 2;
    return bwd_run(&J);
}
