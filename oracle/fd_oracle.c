/*
 * fd_oracle.c -- float64 CPU oracle for split-KV decode attention
 * (FlashDecoding).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded input tensors.
 *
 * Pages followed (cited by title and section):
 *   [FDD]  "FlashDecoding 数学推导"
 *   [ADV4] "adv04: Flash-Decoding（长序列 Decode 切分 + FlashInfer 简介）"
 *   [LSE]  "FlashDecoding 数学推导：传统 m/l/o 方法与 LSE 方法"
 *   [FA1P] "从第一性原理推导 Flash Attention" (its merge lemma, §3.2; paged
 *          KV, §7.1)
 *
 * Everything is computed in IEEE double with plain loops in index order; no
 * blocking, no fusion, no reordering beyond what the cited formulas state.
 * Inputs are read bit-exactly: fp16 and bf16 values widen to double without
 * rounding (decoders below are written from the IEEE-754 binary16 definition
 * and from bf16 being the top half of a binary32).
 *
 * Layouts (all contiguous, row-major):
 *   q   [B, H, d]          K, V [B, H, N, d]       lens [B] (NULL => all N)
 *   out [B, H, d] double   lse  [B, H] double      partials [B, H, P, ...]
 *
 * Readings of the pages that the oracle fixes (each also listed in the
 * design notes):
 *   - lse is the natural-log sum-exp of the *scaled* scores.
 *   - a sequence of length 0 gives out = 0, lse = -inf.
 *   - partial o is stored normalised (divided by its own l), as in [FDD]
 *     §2.4.1 and [LSE] §2.2.1; an empty split is (o=0, m=-inf, l=0,
 *     S=-inf) and every merge gives it weight 0 explicitly (no epsilon).
 *   - the explicit-split partition is [ADV4] §4: chunk = ceil(n / P),
 *     split p covers [p*chunk, min((p+1)*chunk, n)), empty if it starts at
 *     or beyond n.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 };

/* ------------------------------------------------------------------ */
/* element decoders                                                    */
/* ------------------------------------------------------------------ */

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  exponent 0 => subnormal fraction * 2^-24; exponent 31 => inf/nan;
 * otherwise (1024 + fraction) * 2^(exponent - 25). */
double or_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bf16 is the upper 16 bits of an IEEE binary32. */
double or_bf16_to_double(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities; S.1111.111 is NaN.  exponent 0
 * => subnormal mantissa * 2^-9; otherwise (8 + mantissa) * 2^(exponent - 10). */
double or_e4m3_to_double(uint8_t x)
{
    int sign = (x >> 7) & 1;
    int e = (x >> 3) & 0xf;
    int m = x & 0x7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

static double load_elem(const void *base, size_t idx, int dtype)
{
    if (dtype == OR_E4M3)
        return or_e4m3_to_double(((const uint8_t *)base)[idx]);
    if (dtype == OR_F32) {
        float f;
        memcpy(&f, (const char *)base + idx * 4, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + idx * 2, 2);
    return dtype == OR_F16 ? or_f16_to_double(h) : or_bf16_to_double(h);
}

/* Bulk decode, exposed so the tests can pin the decoders exhaustively. */
void or_decode(int dtype, const void *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = load_elem(src, (size_t)i, dtype);
}

/* ------------------------------------------------------------------ */
/* shared argument bundle and a tiny thread pool over (b, h) pairs     */
/* ------------------------------------------------------------------ */

typedef struct {
    const void *q, *k, *v;
    const int32_t *lens;
    int B, H, N, d, dtype, P;
    int kvdtype;                       /* element type of K and V            */
    int G;                             /* query heads per K/V head (>= 1)    */
    const float *k_scale, *v_scale;    /* per-(b,h) dequantisation, or NULL  */
    double scale;
    double *out, *lse;                       /* full attention          */
    double *o_part, *m_part, *l_part, *s_part; /* per-split partials     */
    int nthreads, tid;
} job_t;

typedef void (*pair_fn)(const job_t *, int b, int h);

typedef struct {
    const job_t *job;
    pair_fn fn;
    int tid, nthreads;
} worker_t;

static void *worker_main(void *arg)
{
    const worker_t *w = (const worker_t *)arg;
    int64_t total = (int64_t)w->job->B * w->job->H;
    for (int64_t bh = w->tid; bh < total; bh += w->nthreads)
        w->fn(w->job, (int)(bh / w->job->H), (int)(bh % w->job->H));
    return NULL;
}

static int run_pairs(const job_t *job, pair_fn fn, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;
    worker_t *ws = (worker_t *)calloc((size_t)nthreads, sizeof(worker_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!ws || !th) {
        free(ws);
        free(th);
        return -1;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        ws[t].job = job;
        ws[t].fn = fn;
        ws[t].tid = t;
        ws[t].nthreads = nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker_main, &ws[t]) != 0)
            break;
        started = t;
    }
    /* threads that failed to start have their share done here */
    for (int t = started + 1; t < nthreads; ++t)
        worker_main(&ws[t]);
    worker_main(&ws[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    free(ws);
    free(th);
    return 0;
}

static int seq_len(const job_t *j, int b)
{
    int n = j->lens ? j->lens[b] : j->N;
    if (n < 0)
        n = 0;
    if (n > j->N)
        n = j->N;
    return n;
}

/* a K or V element: the stored value, times its (b,h) scale when one is given */
static double kv_elem(const job_t *j, const void *base, size_t idx, const float *sc, size_t bh)
{
    double x = load_elem(base, idx, j->kvdtype);
    return sc ? (double)sc[bh] * x : x;
}

/* the K/V head of query head h: heads come in groups of G sharing one */
static size_t kv_row(const job_t *j, int b, int h)
{
    int g = j->G > 1 ? j->G : 1;
    return (size_t)b * (size_t)(j->H / g) + (size_t)(h / g);
}

/* score s_j = scale * sum_i q_i K_{j,i}   ([FDD] §2.2, [LSE] §2.1.1) */
static double score(const job_t *j, int b, int h, int t)
{
    size_t bh = (size_t)b * j->H + h;
    size_t kvh = kv_row(j, b, h);
    size_t qb = bh * j->d;
    size_t kb = (kvh * j->N + t) * j->d;
    double acc = 0.0;
    for (int i = 0; i < j->d; ++i)
        acc += load_elem(j->q, qb + i, j->dtype) * kv_elem(j, j->k, kb + i, j->k_scale, kvh);
    return j->scale * acc;
}

/*
 * Direct (two-pass) softmax attention over tokens [lo, hi) of one (b, h):
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  o = sum_j exp(s_j - m) V_j / l
 * This is the per-tile "direct form" of [FDD] §2.4.1 (and [LSE] §2.2.1);
 * with [lo, hi) = [0, n) it is full attention, [LSE] §2.1.1 with the
 * max-shift of [FDD] §2.3.1.  Returns l (0 for an empty range).
 */
static double direct_range(const job_t *j, int b, int h, int lo, int hi,
                           double *o, double *m_out, double *s_scratch)
{
    int d = j->d;
    for (int i = 0; i < d; ++i)
        o[i] = 0.0;
    if (lo >= hi) {
        *m_out = -INFINITY;
        return 0.0;
    }
    double m = -INFINITY;
    for (int t = lo; t < hi; ++t) {
        s_scratch[t - lo] = score(j, b, h, t);
        if (s_scratch[t - lo] > m)
            m = s_scratch[t - lo];
    }
    double l = 0.0;
    size_t kvh = kv_row(j, b, h);
    size_t vb = (kvh * j->N) * d;
    for (int t = lo; t < hi; ++t) {
        double w = exp(s_scratch[t - lo] - m);
        l += w;
        for (int i = 0; i < d; ++i)
            o[i] += w * kv_elem(j, j->v, vb + (size_t)t * d + i, j->v_scale, kvh);
    }
    for (int i = 0; i < d; ++i)
        o[i] /= l;
    *m_out = m;
    return l;
}

static void attention_pair(const job_t *j, int b, int h)
{
    int n = seq_len(j, b);
    size_t bh = (size_t)b * j->H + h;
    double *o = j->out + bh * j->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m;
    double l = direct_range(j, b, h, 0, n, o, &m, s);
    free(s);
    /* lse = m + ln l ([LSE] §2.3.2); empty sequence => -inf */
    if (j->lse)
        j->lse[bh] = (l > 0.0) ? m + log(l) : -INFINITY;
}

/*
 * Full, unsplit single-query attention for every (b, h):
 *   out = softmax(scale * q K^T) V,  lse = ln sum_j exp(scale * q.K_j).
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int or_attention(const void *q, const void *k, const void *v, const int32_t *lens,
                 int B, int H, int N, int d, int dtype, double scale,
                 double *out, double *lse, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || dtype < 0 || dtype > 2 || !out)
        return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.k = k; j.v = v; j.lens = lens;
    j.B = B; j.H = H; j.N = N; j.d = d; j.dtype = dtype; j.kvdtype = dtype;
    j.scale = scale; j.out = out; j.lse = lse;
    return run_pairs(&j, attention_pair, nthreads);
}

/*
 * Grouped-query attention (MQA / GQA, [FA1P] §8): q [B, Hq, d] and K, V
 * [B, Hkv, N, d] with Hq = G * Hkv; query head h attends with K/V head
 * h / G (consecutive query heads share a K/V head).  Everything else is
 * or_attention.  out [B, Hq, d], lse [B, Hq].
 */
int or_attention_gqa(const void *q, const void *k, const void *v, const int32_t *lens,
                     int B, int Hq, int Hkv, int N, int d, int dtype, double scale,
                     double *out, double *lse, int nthreads)
{
    if (B < 0 || Hq < 0 || Hkv <= 0 || Hq % Hkv != 0 || N < 0 || d <= 0 || dtype < 0 ||
        dtype > 2 || !out)
        return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.k = k; j.v = v; j.lens = lens;
    j.B = B; j.H = Hq; j.N = N; j.d = d; j.dtype = dtype; j.kvdtype = dtype;
    j.G = Hq / Hkv;
    j.scale = scale; j.out = out; j.lse = lse;
    return run_pairs(&j, attention_pair, nthreads);
}

/*
 * Full attention over an FP8 (E4M3) KV cache with per-(b,h) scales: the
 * value of K[b,h,t,i] is k_scale[b*H+h] * e4m3(k[b,h,t,i]), likewise V.  The
 * low-precision storage is the "FP8 support" of [FA1P] §6.2 applied to the
 * cache; the attention is exactly or_attention's on those values.  q is
 * f32 / f16 / bf16 (q_dtype).
 */
int or_attention_fp8(const void *q, int q_dtype, const void *k, const void *v,
                     const float *k_scale, const float *v_scale, const int32_t *lens,
                     int B, int H, int N, int d, double scale, double *out, double *lse,
                     int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || q_dtype < 0 || q_dtype > 2 || !out ||
        !k_scale || !v_scale)
        return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.k = k; j.v = v; j.lens = lens;
    j.B = B; j.H = H; j.N = N; j.d = d; j.dtype = q_dtype; j.kvdtype = OR_E4M3;
    j.k_scale = k_scale; j.v_scale = v_scale;
    j.scale = scale; j.out = out; j.lse = lse;
    return run_pairs(&j, attention_pair, nthreads);
}

static void split_pair(const job_t *j, int b, int h)
{
    int n = seq_len(j, b);
    int P = j->P;
    int chunk = (n + P - 1) / P; /* [ADV4] §4: ceil(seq / num_splits) */
    size_t bh = (size_t)b * j->H + h;
    double *s = (double *)malloc(sizeof(double) * (size_t)(chunk > 0 ? chunk : 1));
    for (int p = 0; p < P; ++p) {
        int64_t lo64 = (int64_t)p * chunk;
        int lo = lo64 > n ? n : (int)lo64;
        int hi = (lo + chunk < n) ? lo + chunk : n;
        size_t slot = bh * P + p;
        double m;
        double l = direct_range(j, b, h, lo, hi, j->o_part + slot * j->d, &m, s);
        j->m_part[slot] = m;
        j->l_part[slot] = l;
        if (j->s_part)
            j->s_part[slot] = (l > 0.0) ? m + log(l) : -INFINITY;
    }
    free(s);
}

/*
 * Per-split partials in the partition of [ADV4] §4, each in the direct form
 * of [FDD] §2.4.1: (o normalised, m, l) and S = m + ln l ([LSE] §2.3.2).
 * o_part [B,H,P,d], m_part/l_part/s_part [B,H,P] (s_part may be NULL).
 */
int or_split_partials(const void *q, const void *k, const void *v, const int32_t *lens,
                      int B, int H, int N, int d, int dtype, double scale, int P,
                      double *o_part, double *m_part, double *l_part, double *s_part,
                      int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || P < 1 || dtype < 0 || dtype > 2 ||
        !o_part || !m_part || !l_part)
        return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.k = k; j.v = v; j.lens = lens;
    j.B = B; j.H = H; j.N = N; j.d = d; j.dtype = dtype; j.kvdtype = dtype; j.P = P;
    j.scale = scale;
    j.o_part = o_part; j.m_part = m_part; j.l_part = l_part; j.s_part = s_part;
    return run_pairs(&j, split_pair, nthreads);
}

/* ------------------------------------------------------------------ */
/* paged KV cache                                                      */
/* ------------------------------------------------------------------ */

/*
 * Full attention over a paged KV cache (the block-table indirection of
 * [ADV4] §5 "分页 KV Cache" and [FA1P] §7.1).  Pages are laid out
 * [num_pages, H, page_size, d]; logical token t of sequence b is row
 * t % page_size of head h in physical page block_table[b*max_pages +
 * t/page_size].  lens is required.  The arithmetic is or_attention's on the
 * gathered rows.  Returns -1 on bad arguments or a table entry outside
 * [0, num_pages).
 */
typedef struct {
    const void *q, *kp, *vp;
    const int32_t *table, *lens;
    int B, H, d, ps, maxp, dtype;
    int64_t num_pages;
    double scale;
    double *out, *lse;
    int bad;
} pjob_t;

static size_t paged_row(const pjob_t *j, int b, int h, int t)
{
    int32_t pg = j->table[(int64_t)b * j->maxp + t / j->ps];
    return (((size_t)pg * j->H + h) * j->ps + (size_t)(t % j->ps)) * j->d;
}

static void *paged_worker(void *arg)
{
    pjob_t **pp = (pjob_t **)arg;
    pjob_t *j = pp[0];
    int tid = (int)(intptr_t)pp[1], nth = (int)(intptr_t)pp[2];
    int64_t total = (int64_t)j->B * j->H;
    for (int64_t bh = tid; bh < total; bh += nth) {
        int b = (int)(bh / j->H), h = (int)(bh % j->H);
        int n = j->lens[b];
        if (n < 0)
            n = 0;
        if (n > j->maxp * j->ps)
            n = j->maxp * j->ps;
        double *o = j->out + bh * j->d;
        for (int i = 0; i < j->d; ++i)
            o[i] = 0.0;
        if (n == 0) {
            if (j->lse)
                j->lse[bh] = -INFINITY;
            continue;
        }
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        if (!s) {
            j->bad = 1;
            continue;
        }
        size_t qb = (size_t)bh * j->d;
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            size_t kr = paged_row(j, b, h, t);
            double acc = 0.0;
            for (int i = 0; i < j->d; ++i)
                acc += load_elem(j->q, qb + i, j->dtype) * load_elem(j->kp, kr + i, j->dtype);
            s[t] = j->scale * acc;
            if (s[t] > m)
                m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < n; ++t) {
            double w = exp(s[t] - m);
            size_t vr = paged_row(j, b, h, t);
            l += w;
            for (int i = 0; i < j->d; ++i)
                o[i] += w * load_elem(j->vp, vr + i, j->dtype);
        }
        for (int i = 0; i < j->d; ++i)
            o[i] /= l;
        if (j->lse)
            j->lse[bh] = m + log(l);
        free(s);
    }
    return NULL;
}

int or_attention_paged(const void *q, const void *k_pages, const void *v_pages,
                       const int32_t *block_table, const int32_t *lens, int B, int H, int d,
                       int page_size, int max_pages, int64_t num_pages, int dtype, double scale,
                       double *out, double *lse, int nthreads)
{
    if (B < 0 || H < 0 || d <= 0 || page_size < 1 || max_pages < 0 || num_pages < 0 ||
        dtype < 0 || dtype > 2 || !out || !lens)
        return -1;
    /* every table entry a sequence uses must name an existing page */
    for (int b = 0; b < B; ++b) {
        int n = lens[b] < 0 ? 0 : lens[b];
        if (n > max_pages * page_size)
            n = max_pages * page_size;
        for (int pgi = 0; pgi * page_size < n; ++pgi) {
            int32_t pg = block_table[(int64_t)b * max_pages + pgi];
            if (pg < 0 || pg >= num_pages)
                return -1;
        }
    }
    pjob_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.kp = k_pages; j.vp = v_pages; j.table = block_table; j.lens = lens;
    j.B = B; j.H = H; j.d = d; j.ps = page_size; j.maxp = max_pages; j.dtype = dtype;
    j.num_pages = num_pages; j.scale = scale; j.out = out; j.lse = lse;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    void *(*args)[3] = calloc((size_t)nthreads, sizeof *args);
    if (!th || !args) {
        free(th);
        free(args);
        return -1;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t][0] = &j;
        args[t][1] = (void *)(intptr_t)t;
        args[t][2] = (void *)(intptr_t)nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, paged_worker, args[t]) != 0)
            break;
        started = t;
    }
    for (int t = started + 1; t < nthreads; ++t)
        paged_worker(args[t]);
    paged_worker(args[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(args);
    return j.bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* merges of partials (all per (b,h) row of P partials)                */
/* ------------------------------------------------------------------ */

/*
 * m/l/o global merge, [FDD] §2.4.2 steps 1-3 (= [LSE] §2.2.2):
 *   m_g = max_p m_p,  l_g = sum_p exp(m_p - m_g) l_p,
 *   o   = sum_p exp(m_p - m_g) l_p o_p / l_g,   lse = m_g + ln l_g.
 * Splits with l_p == 0 (empty) are skipped: weight 0.
 */
void or_combine_mlo(const double *o_part, const double *m_part, const double *l_part,
                    int64_t rows, int P, int d, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *o = o_part + r * P * d, *m = m_part + r * P, *l = l_part + r * P;
        double mg = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (l[p] > 0.0 && m[p] > mg)
                mg = m[p];
        double lg = 0.0;
        for (int p = 0; p < P; ++p)
            if (l[p] > 0.0)
                lg += exp(m[p] - mg) * l[p];
        for (int i = 0; i < d; ++i) {
            double num = 0.0;
            for (int p = 0; p < P; ++p)
                if (l[p] > 0.0)
                    num += exp(m[p] - mg) * l[p] * o[(int64_t)p * d + i];
            out[r * d + i] = (lg > 0.0) ? num / lg : 0.0;
        }
        if (lse)
            lse[r] = (lg > 0.0) ? mg + log(lg) : -INFINITY;
    }
}

/*
 * LSE global merge, [LSE] §2.3.4:
 *   S_g = ln sum_p exp(S_p)  (evaluated with the max shift of its safe-LSE
 *   card: S_max + ln sum_p exp(S_p - S_max)),
 *   o   = sum_p exp(S_p - S_g) o_p.
 * Splits with S_p == -inf (empty) are skipped: weight 0.
 */
void or_combine_lse(const double *o_part, const double *s_part,
                    int64_t rows, int P, int d, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *o = o_part + r * P * d, *S = s_part + r * P;
        double smax = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (S[p] > smax)
                smax = S[p];
        double sum = 0.0;
        for (int p = 0; p < P; ++p)
            if (S[p] != -INFINITY)
                sum += exp(S[p] - smax);
        double sg = (sum > 0.0) ? smax + log(sum) : -INFINITY;
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int p = 0; p < P; ++p)
                if (S[p] != -INFINITY)
                    acc += exp(S[p] - sg) * o[(int64_t)p * d + i];
            out[r * d + i] = acc;
        }
        if (lse)
            lse[r] = sg;
    }
}

/*
 * Sequential fold with the two-term operator (+) of [LSE] §2.3.5, evaluated
 * in the safe form of [LSE] §3.2.1 stage 2:
 *   S_new = S_max + log1p(exp(S_min - S_max)),
 *   o_new = o_acc exp(S_acc - S_new) + o_i exp(S_i - S_new).
 * The accumulator starts empty (S = -inf); an empty operand leaves the other
 * unchanged.
 */
void or_merge_lse_sequential(const double *o_part, const double *s_part,
                             int64_t rows, int P, int d, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double *o = out + r * d;
        double S = -INFINITY;
        for (int i = 0; i < d; ++i)
            o[i] = 0.0;
        for (int p = 0; p < P; ++p) {
            double Si = s_part[r * P + p];
            const double *oi = o_part + (r * P + p) * d;
            if (Si == -INFINITY)
                continue;
            if (S == -INFINITY) {
                S = Si;
                for (int i = 0; i < d; ++i)
                    o[i] = oi[i];
                continue;
            }
            double smax = S > Si ? S : Si, smin = S > Si ? Si : S;
            double Sn = smax + log1p(exp(smin - smax));
            double wa = exp(S - Sn), wi = exp(Si - Sn);
            for (int i = 0; i < d; ++i)
                o[i] = o[i] * wa + oi[i] * wi;
            S = Sn;
        }
        if (lse)
            lse[r] = S;
    }
}

/*
 * Pairwise tree reduction of unnormalised (O, M, L) triples, the merge lemma
 * of [FA1P] §3.2 applied level by level as in [LSE] §3.1.3:
 *   M = max(M1, M2), L = e^{M1-M} L1 + e^{M2-M} L2, O = e^{M1-M} O1 + e^{M2-M} O2,
 * an odd element passing up unchanged; the result is O / L.  The inputs are
 * normalised partials, so O_p = l_p o_p is formed first.
 */
int or_merge_mlo_tree(const double *o_part, const double *m_part, const double *l_part,
                      int64_t rows, int P, int d, double *out, double *lse)
{
    double *O = (double *)malloc(sizeof(double) * (size_t)P * d);
    double *M = (double *)malloc(sizeof(double) * (size_t)P);
    double *L = (double *)malloc(sizeof(double) * (size_t)P);
    if (!O || !M || !L) {
        free(O); free(M); free(L);
        return -1;
    }
    for (int64_t r = 0; r < rows; ++r) {
        for (int p = 0; p < P; ++p) {
            double lp = l_part[r * P + p];
            M[p] = m_part[r * P + p];
            L[p] = lp;
            for (int i = 0; i < d; ++i)
                O[(int64_t)p * d + i] = (lp > 0.0) ? lp * o_part[(r * P + p) * d + i] : 0.0;
        }
        int n = P;
        while (n > 1) {
            int w = 0;
            for (int a = 0; a < n; a += 2, ++w) {
                if (a + 1 >= n) {
                    M[w] = M[a];
                    L[w] = L[a];
                    for (int i = 0; i < d; ++i)
                        O[(int64_t)w * d + i] = O[(int64_t)a * d + i];
                    continue;
                }
                double m1 = M[a], m2 = M[a + 1], l1 = L[a], l2 = L[a + 1];
                double mn = m1 > m2 ? m1 : m2;
                /* an empty side (L == 0, M == -inf) gets weight 0 explicitly */
                double c1 = (l1 > 0.0) ? exp(m1 - mn) : 0.0;
                double c2 = (l2 > 0.0) ? exp(m2 - mn) : 0.0;
                M[w] = mn;
                L[w] = c1 * l1 + c2 * l2;
                for (int i = 0; i < d; ++i)
                    O[(int64_t)w * d + i] = c1 * O[(int64_t)a * d + i] + c2 * O[(int64_t)(a + 1) * d + i];
            }
            n = w;
        }
        for (int i = 0; i < d; ++i)
            out[r * d + i] = (L[0] > 0.0) ? O[i] / L[0] : 0.0;
        if (lse)
            lse[r] = (L[0] > 0.0) ? M[0] + log(L[0]) : -INFINITY;
    }
    free(O); free(M); free(L);
    return 0;
}

/* ------------------------------------------------------------------ */
/* the recurrences themselves (small cases, for the worked examples)   */
/* ------------------------------------------------------------------ */

/*
 * Online softmax (m, d) recurrence of [FDD] §2.3.2 over x[0..n):
 *   m_1 = x_1, d_1 = 1;  m_j = max(m_{j-1}, x_j),
 *   d_j = d_{j-1} exp(m_{j-1} - m_j) + exp(x_j - m_j).
 * m_steps / d_steps (may be NULL) receive every intermediate state.
 */
void or_online_softmax(const double *x, int n, double *m_steps, double *d_steps,
                       double *m_out, double *d_out)
{
    double m = -INFINITY, dd = 0.0;
    for (int j = 0; j < n; ++j) {
        if (j == 0) {
            m = x[0];
            dd = 1.0;
        } else {
            double mn = x[j] > m ? x[j] : m;
            dd = dd * exp(m - mn) + exp(x[j] - mn);
            m = mn;
        }
        if (m_steps)
            m_steps[j] = m;
        if (d_steps)
            d_steps[j] = dd;
    }
    *m_out = m;
    *d_out = dd;
}

/*
 * Incremental per-token update of [FDD] §2.4.1 ("增量更新") over the given
 * scores s[0..n) and value rows V[n][d] (double):
 *   m_1 = s_1, l_1 = 1, o_1 = V_1;
 *   m_j = max(m_{j-1}, s_j),  l_j = l_{j-1} e^{m_{j-1}-m_j} + e^{s_j-m_j},
 *   o_j = (l_{j-1} e^{m_{j-1}-m_j} o_{j-1} + e^{s_j-m_j} V_j) / l_j.
 * Step states are written to m_steps[n], l_steps[n], o_steps[n][d] if
 * non-NULL; the final (m, l, o) to the outputs.
 */
void or_tile_incremental(const double *s, const double *V, int n, int d,
                         double *m_steps, double *l_steps, double *o_steps,
                         double *m_out, double *l_out, double *o_out)
{
    double m = -INFINITY, l = 0.0;
    for (int i = 0; i < d; ++i)
        o_out[i] = 0.0;
    for (int j = 0; j < n; ++j) {
        if (j == 0) {
            m = s[0];
            l = 1.0;
            for (int i = 0; i < d; ++i)
                o_out[i] = V[i];
        } else {
            double mn = s[j] > m ? s[j] : m;
            double carry = l * exp(m - mn);
            double w = exp(s[j] - mn);
            double ln = carry + w;
            for (int i = 0; i < d; ++i)
                o_out[i] = (carry * o_out[i] + w * V[(int64_t)j * d + i]) / ln;
            m = mn;
            l = ln;
        }
        if (m_steps)
            m_steps[j] = m;
        if (l_steps)
            l_steps[j] = l;
        if (o_steps)
            for (int i = 0; i < d; ++i)
                o_steps[(int64_t)j * d + i] = o_out[i];
    }
    *m_out = m;
    *l_out = l;
}
