/*
 * Plain fp64 CPU oracle for the CSA / HCA attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the layer computes.  Only the test suite, the smoke check
 * and the bench's CPU-baseline leg load it; the product library never does,
 * and it shares no code, header or table with the CUDA path.
 *
 * Sources (web pages about the DeepSeek-V4 report):
 *   [Book]  "DeepSeek-V4" book (slop-6tp.pages.dev/papers-html/dsv4),
 *           ch.5 "How CSA Compresses Memory", ch.6 "How CSA Selects and Reads
 *           Memory", ch.7 "HCA, Local Attention, and Position".
 *   [Notes] "DeepSeek-V4: Making Million-Token Context an Architectural
 *           Problem", Key design 1 (CSA compression and index-score
 *           equations), Key design 2 (HCA compression equation).
 *   [Expl]  "DeepSeek-V4" explainer (aiany.app): "every m consecutive tokens".
 *
 * Every routine is the plain definition, evaluated directly in double
 * precision, in the order the definition states it.  Inputs arrive in their
 * storage dtype and are widened exactly to double on read:
 *   dtype 0 = double, 1 = float, 2 = bfloat16 bit patterns (uint16).
 *
 * Readings fixed where the pages are silent (all restated here):
 *   - single-branch compression (overlap = 0): the block i is positions
 *     m*i .. m*i+m-1; two-branch (overlap = 1) adds the b branch over block
 *     i-1, which for i = 0 has zero content and logit -inf.
 *   - entry j is visible to the query at position t iff (j+1)*m <= t+1.
 *   - the window is the raw rows at positions max(0, t-n_win+1) .. t.
 *   - RoPE rotates adjacent pairs (c-r+2i, c-r+2i+1) of the last r dims by
 *     angle p * theta^(-2i/r); a compressed entry sits at position (j+1)*m-1;
 *     stored entries and stored raw rows carry their rotation (it is applied
 *     when the cache is written), queries are rotated at t inside attention,
 *     and the output's rotary dims are rotated back by -t when derotate = 1.
 *   - the indexer uses no RoPE and no scale.
 *   - top-k keeps all visible entries when there are at most k; otherwise
 *     the k best by (score descending, index ascending); output ascending.
 *   - logit scale 1/sqrt(c) unless given; sink logit only in the denominator.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- inputs */

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double ld(const void *p, int dt, int64_t i)
{
    switch (dt) {
    case 0: return ((const double *)p)[i];
    case 1: return (double)((const float *)p)[i];
    default: return bf16_to_double(((const uint16_t *)p)[i]);
    }
}

/* Round a double to the storage dtype, nearest with ties to even, and
 * return the rounded value as a double.  bf16 keeps 8 significant bits. */
static double round_to(double x, int dt)
{
    if (dt == 0 || x == 0.0 || !isfinite(x))
        return x;
    if (dt == 1)
        return (double)(float)x;            /* C conversion: nearest-even */
    int e = ilogb(x);                        /* |x| in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;                            /* bf16 subnormal spacing 2^-133 */
    double ulp = ldexp(1.0, e - 7);
    double r = nearbyint(x / ulp) * ulp;     /* default mode: ties to even */
    if (fabs(r) > 3.3895313892515355e38)     /* beyond bf16 max */
        r = copysign(INFINITY, x);
    return r;
}

/* ------------------------------------------------------------------ RoPE */

/* [Book] ch.7 "Partial rotary position embeddings": rotate the last r
 * coordinates of a length-c vector by position p, pairs (2i, 2i+1). */
void orc_rope(double *x, int c, int r, double theta, double p)
{
    for (int i = 0; i < r / 2; i++) {
        double w = pow(theta, -2.0 * i / (double)r);
        double a = p * w;
        double cs = cos(a), sn = sin(a);
        double *v = x + (c - r) + 2 * i;
        double x0 = v[0], x1 = v[1];
        v[0] = x0 * cs - x1 * sn;
        v[1] = x0 * sn + x1 * cs;
    }
}

/* Stored raw rows: rotate row l at position pos0 + l, then round. */
void orc_rope_rows(int dt_in, const void *x, int64_t L, int c, int r, double theta,
                   int64_t pos0, int dt_out, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t l = 0; l < L; l++) {
        double *o = out + l * c;
        for (int ch = 0; ch < c; ch++)
            o[ch] = ld(x, dt_in, l * c + ch);
        orc_rope(o, c, r, theta, (double)(pos0 + l));
        for (int ch = 0; ch < c; ch++)
            o[ch] = round_to(o[ch], dt_out);
    }
}

/* ----------------------------------------------------------- compression */

/*
 * [Notes] Key design 1 (two-branch equation) and Key design 2 (HCA
 * equation); [Book] ch.5 "One weight distribution per coordinate" and
 * "Which positions enter a compressed block"; [Expl] "every m consecutive
 * tokens".  For each complete block i and channel ch, the weights are a
 * softmax over the block's source positions of (logit + per-slot bias),
 * separately per channel; the entry is the weighted sum of the content.
 *
 * One sequence: C, Z [n, c]; bias [m, c]; overlap adds Cb, Zb [n, c],
 * biasb [m, c].  Output [n/m, c]: rotated by RoPE at the block's last
 * position (r = 0 for none), then rounded to dt_out.
 */
void orc_compress(int dt, const void *C, const void *Z, const void *bias, int dt_bias,
                  const void *Cb, const void *Zb, const void *biasb,
                  int64_t n, int c, int m, int overlap,
                  int r, double theta, int dt_out, double *out)
{
    int64_t E = n / m;
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * 2 * m);
        double *v = (double *)malloc(sizeof(double) * 2 * m);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < E; i++) {
            double *o = out + i * c;
            for (int ch = 0; ch < c; ch++) {
                int ns = 0;
                for (int s = 0; s < m; s++) {
                    int64_t row = (int64_t)m * i + s;
                    a[ns] = ld(Z, dt, row * c + ch) + ld(bias, dt_bias, (int64_t)s * c + ch);
                    v[ns] = ld(C, dt, row * c + ch);
                    ns++;
                }
                if (overlap) {
                    for (int s = 0; s < m; s++) {
                        if (i == 0) {             /* no previous block */
                            a[ns] = -INFINITY;
                            v[ns] = 0.0;
                        } else {
                            int64_t row = (int64_t)m * (i - 1) + s;
                            a[ns] = ld(Zb, dt, row * c + ch) + ld(biasb, dt_bias, (int64_t)s * c + ch);
                            v[ns] = ld(Cb, dt, row * c + ch);
                        }
                        ns++;
                    }
                }
                double mx = -INFINITY;
                for (int s = 0; s < ns; s++)
                    if (a[s] > mx) mx = a[s];
                double den = 0.0, num = 0.0;
                for (int s = 0; s < ns; s++) {
                    double e = exp(a[s] - mx);
                    den += e;
                    num += e * v[s];
                }
                o[ch] = num / den;
            }
            if (r > 0)
                orc_rope(o, c, r, theta, (double)((i + 1) * (int64_t)m - 1));
            for (int ch = 0; ch < c; ch++)
                o[ch] = round_to(o[ch], dt_out);
        }
        free(a);
        free(v);
    }
}

/* ------------------------------------------------------------ visibility */

/* Entry j is visible at query position t iff (j+1)*m <= t+1. */
int64_t orc_visible(int64_t t, int m, int64_t E)
{
    int64_t v = (t + 1) / m;
    if (v > E) v = E;
    if (v < 0) v = 0;
    return v;
}

/* --------------------------------------------------------------- indexer */

/*
 * [Notes] Key design 1, index score: I[t,j] = sum_h w[t,h] * ReLU(qI[t,h] . kI[j]);
 * [Book] ch.6 "The index score".  Invisible entries get -inf.
 * qI [T, hI, dI], w [T, hI], kI [E, dI], q_pos [T] -> scores [T, E].
 */
void orc_index_scores(int dt_q, const void *qI, int dt_w, const void *w, const int64_t *q_pos,
                      int64_t T, int hI, int dI,
                      int dt_k, const void *kI, int64_t E, int m, double *scores)
{
    double *qt = (double *)malloc(sizeof(double) * hI * dI);
    double *wt = (double *)malloc(sizeof(double) * hI);
    for (int64_t t = 0; t < T; t++) {
        for (int i = 0; i < hI * dI; i++)
            qt[i] = ld(qI, dt_q, t * hI * dI + i);
        for (int h = 0; h < hI; h++)
            wt[h] = ld(w, dt_w, t * hI + h);
        int64_t nv = orc_visible(q_pos[t], m, E);
#pragma omp parallel
        {
            double *kj = (double *)malloc(sizeof(double) * dI);
#pragma omp for schedule(static)
            for (int64_t j = 0; j < E; j++) {
                double s;
                if (j >= nv) {
                    s = -INFINITY;
                } else {
                    for (int d = 0; d < dI; d++)
                        kj[d] = ld(kI, dt_k, j * dI + d);
                    s = 0.0;
                    for (int h = 0; h < hI; h++) {
                        double dot = 0.0;
                        for (int d = 0; d < dI; d++)
                            dot += qt[h * dI + d] * kj[d];
                        double relu = dot > 0.0 ? dot : 0.0;
                        s += wt[h] * relu;
                    }
                }
                scores[t * E + j] = s;
            }
            free(kj);
        }
    }
    free(qt);
    free(wt);
}

/* ----------------------------------------------------------------- top-k */

typedef struct { double s; int64_t j; } orc_cand;

static int orc_cand_cmp(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    if (a->s > b->s) return -1;          /* score descending */
    if (a->s < b->s) return 1;
    return (a->j < b->j) ? -1 : (a->j > b->j);   /* ties: lower index first */
}

static int orc_i32_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * [Notes] Key design 1, C_t = TopK_k(I[t,:]); [Book] ch.6 "Top-k is a budget
 * over compressed entries": with at most k visible entries all are kept.
 * scores [T, E] -> idx [T, k] ascending, -1 padded; cnt [T].
 */
void orc_topk(const double *scores, const int64_t *q_pos, int64_t T, int64_t E, int m, int k,
              int32_t *idx, int32_t *cnt)
{
#pragma omp parallel
    {
        orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (E > 0 ? E : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; t++) {
            int64_t nv = orc_visible(q_pos[t], m, E);
            int32_t *o = idx + t * k;
            int64_t keep;
            if (nv <= k) {
                for (int64_t j = 0; j < nv; j++)
                    o[j] = (int32_t)j;
                keep = nv;
            } else {
                for (int64_t j = 0; j < nv; j++) {
                    double s = scores[t * E + j];
                    cand[j].s = (s == 0.0) ? 0.0 : s;     /* -0 ties with +0 */
                    cand[j].j = j;
                }
                qsort(cand, (size_t)nv, sizeof(orc_cand), orc_cand_cmp);
                for (int i = 0; i < k; i++)
                    o[i] = (int32_t)cand[i].j;
                qsort(o, (size_t)k, sizeof(int32_t), orc_i32_cmp);
                keep = k;
            }
            for (int64_t i = keep; i < k; i++)
                o[i] = -1;
            cnt[t] = (int32_t)keep;
        }
        free(cand);
    }
}

/* ------------------------------------------------------------- attention */

/*
 * Shared-KV MQA core attention with window and sink, for one sequence.
 * [Book] ch.6 "Shared key-value MQA"; ch.7 "The sliding window", "Partial
 * rotary position embeddings", "Why the output is de-rotated", "Attention
 * sinks"; [Notes] Key design 1 and 2.
 *
 * For query t and head h, over the set S = selected (idx != NULL) or all
 * visible (idx == NULL) compressed entries u_j = kvc[j], plus the window
 * rows u_p = kv_raw[p - raw_pos0] for p in max(0, t-n_win+1) .. t:
 *   q~ = RoPE(q[t,h], t);  l = scale * (q~ . u)
 *   out = sum e^l u / (e^{sink_h} + sum e^l)
 *   derotate: out[rotary dims] <- RoPE(out, -t)
 *   lse = log(e^{sink_h} + sum e^l)
 * q [T, H, c]; kvc [E, c]; idx [T, k]; kv_raw [L, c]; sink [H].
 * Returns the number of window positions that were missing from kv_raw
 * (they are skipped; 0 means the input covered every window).
 */
int64_t orc_attend(int dt_q, const void *q, const int64_t *q_pos, int64_t T, int H, int c,
                   int dt_kv, const void *kvc, int64_t E, int m,
                   const int32_t *idx, int k,
                   const void *kv_raw, int64_t L, int64_t raw_pos0, int n_win,
                   int dt_sink, const void *sink, int r, double theta, double scale, int derotate,
                   double *out, double *lse)
{
    int64_t missing = 0;
    if (scale == 0.0)
        scale = 1.0 / sqrt((double)c);
#pragma omp parallel reduction(+ : missing)
    {
        int64_t cap = (idx ? k : E) + (n_win > 0 ? n_win : 0) + 1;
        double *buf = (double *)malloc(sizeof(double) * cap * c);
        double *qt = (double *)malloc(sizeof(double) * c);
        double *lg = (double *)malloc(sizeof(double) * cap);
        double *acc = (double *)malloc(sizeof(double) * c);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; t++) {
            int64_t tp = q_pos[t];
            int64_t ne = 0;
            /* compressed entries */
            if (idx) {
                for (int i = 0; i < k; i++) {
                    int32_t j = idx[t * k + i];
                    if (j < 0) continue;
                    for (int ch = 0; ch < c; ch++)
                        buf[ne * c + ch] = ld(kvc, dt_kv, (int64_t)j * c + ch);
                    ne++;
                }
            } else {
                int64_t nv = orc_visible(tp, m, E);
                for (int64_t j = 0; j < nv; j++) {
                    for (int ch = 0; ch < c; ch++)
                        buf[ne * c + ch] = ld(kvc, dt_kv, j * c + ch);
                    ne++;
                }
            }
            /* window rows */
            int64_t p0 = tp - n_win + 1;
            if (p0 < 0) p0 = 0;
            for (int64_t p = p0; p <= tp && n_win > 0; p++) {
                int64_t row = p - raw_pos0;
                if (row < 0 || row >= L) { missing++; continue; }
                for (int ch = 0; ch < c; ch++)
                    buf[ne * c + ch] = ld(kv_raw, dt_kv, row * c + ch);
                ne++;
            }
            for (int h = 0; h < H; h++) {
                for (int ch = 0; ch < c; ch++)
                    qt[ch] = ld(q, dt_q, (t * H + h) * (int64_t)c + ch);
                orc_rope(qt, c, r, theta, (double)tp);
                double z = ld(sink, dt_sink, h);
                double mx = z;
                for (int64_t e = 0; e < ne; e++) {
                    double d = 0.0;
                    for (int ch = 0; ch < c; ch++)
                        d += qt[ch] * buf[e * c + ch];
                    lg[e] = scale * d;
                    if (lg[e] > mx) mx = lg[e];
                }
                double den = (z == -INFINITY) ? 0.0 : exp(z - mx);
                for (int ch = 0; ch < c; ch++)
                    acc[ch] = 0.0;
                for (int64_t e = 0; e < ne; e++) {
                    double p = exp(lg[e] - mx);
                    den += p;
                    for (int ch = 0; ch < c; ch++)
                        acc[ch] += p * buf[e * c + ch];
                }
                double *o = out + (t * H + h) * (int64_t)c;
                for (int ch = 0; ch < c; ch++)
                    o[ch] = den > 0.0 ? acc[ch] / den : 0.0;
                if (derotate)
                    orc_rope(o, c, r, theta, -(double)tp);
                if (lse)
                    lse[t * H + h] = den > 0.0 ? mx + log(den) : -INFINITY;
            }
        }
        free(buf);
        free(qt);
        free(lg);
        free(acc);
    }
    return missing;
}

/* Round an array to a storage dtype in place (a stored tensor's values). */
void orc_round(double *x, int64_t n, int dt)
{
    for (int64_t i = 0; i < n; i++)
        x[i] = round_to(x[i], dt);
}
