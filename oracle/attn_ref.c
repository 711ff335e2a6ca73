/*
 * attn_ref.c -- plain, slow, single-threaded fp64 reference of the fused FP8
 * attention forward.  TEST INFRASTRUCTURE ONLY: the unit tests, the smoke check
 * and the CPU-baseline leg of the benchmark call it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * What it computes (one query row i of request b, query head h):
 *
 *   g      = h / (Hq / Hkv)                      GQA: contiguous groups of q-heads
 *   s_j    = softmax_scale * dq[b,g] * dk[b,g] * sum_t Q[i,t] K[j,t]      (j visible)
 *   m      = max( max_j s_j , sink[h] if a sink is given )
 *   Z      = sum_j exp(s_j - m)  + ( exp(sink[h] - m) if a sink is given )
 *   O[i,:] = dv[b,g] * sum_j exp(s_j - m) V[j,:] / Z
 *   LSE    = m + ln Z
 *
 * Sources (page title, section):
 *  - "PyTorch ... FlashAttention-4 MXFP8", section 2.1 Attention Forward:
 *    S = Q K^T, P = softmax(S), O = P V.
 *  - "[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for Hopper", Design,
 *    "Descales": the q/k descales multiply the softmax scale, the v descale
 *    multiplies the normalised output; each is 0-d or (batch, kv_heads).
 *  - same page, "Supported": causal, sliding (left) window, varlen, paged K/V,
 *    PackGQA, learnable sink.
 *  - "tml-fa4 PR #4" Summary: the 2^8 P bias cancels in the O normalisation and is
 *    removed from the LSE, so the LSE reported is that of the unbiased scores.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - causal masking is bottom-right aligned: key j is visible to query i when
 *    j <= i + (Lk - Lq);
 *  - a left window w >= 0 keeps keys j >= i + (Lk - Lq) - w;
 *  - the sink is a natural-log logit in the units of the scaled scores; it adds
 *    exp(sink) to the denominator only (no value row) and is part of the LSE;
 *  - a row with no visible key and no sink has O = 0 and LSE = -inf; with a sink,
 *    O = 0 and LSE = sink.
 *
 * Inputs are the raw E4M3 codes; they are decoded exactly to fp64 here from the
 * format definition (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite magnitude 448).
 *
 * Build-time mutants (ORACLE_MUTANT=n) plant one plausible mistake each; the
 * pin tests compile them and check that some pin fails.  The default build has
 * ORACLE_MUTANT undefined (0) and no mistake.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* E4M3 ("fn" variant, no infinities) decoded from its bit fields. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0) {
        /* subnormal: 0.mmm * 2^(1 - 7) */
        mag = ldexp((double)mant / 8.0, -6);
    } else {
#if ORACLE_MUTANT == 1
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 8); /* wrong exponent bias */
#else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
#endif
    }
    return sign ? -mag : mag;
}

typedef struct {
    int32_t B, Hq, Hkv, D, DV;
    const uint8_t *q;        /* [total_q][Hq][D] E4M3 codes                         */
    const uint8_t *k;        /* contiguous: [total_k][Hkv][D]; paged: [pages][page_size][Hkv][D] */
    const uint8_t *v;        /* same as k with DV                                   */
    const int32_t *cu_q;     /* [B+1] query-token prefix sums                       */
    const int32_t *cu_k;     /* [B+1] key prefix sums (token offsets, or lengths when paged) */
    const int32_t *block_table; /* NULL, or [B][max_pages] page ids                 */
    int32_t max_pages, page_size;
    const double *dq, *dk, *dv; /* [B][Hkv] each                                    */
    const double *sink;      /* [Hq] or NULL                                        */
    double softmax_scale;
    int32_t causal, window_left;
    int64_t n_rows;          /* < 0: every (token, head); else the listed pairs     */
    const int64_t *rows_tok;
    const int32_t *rows_head;
} oracle_problem;

#if ORACLE_MUTANT == 10
/* a + b rounded to fp32 toward zero (exact sum in fp64, then the fp32 neighbour of
   smaller magnitude) */
static float truncf_add(float a, float b)
{
    double e = (double)a + (double)b;
    float f = (float)e;
    if (fabs((double)f) > fabs(e))
        f = nextafterf(f, 0.0f);
    return f;
}
#endif

/* Pointer to key row j (0-based within request b) for kv-head g. */
static const uint8_t *key_row(const oracle_problem *p, const uint8_t *base, int width,
                              int b, int g, int64_t j)
{
    int64_t tok;
    if (p->block_table) {
        int64_t page = p->block_table[(int64_t)b * p->max_pages + j / p->page_size];
        tok = page * p->page_size + j % p->page_size;
    } else {
        tok = (int64_t)p->cu_k[b] + j;
    }
    return base + (tok * p->Hkv + g) * (int64_t)width;
}

static int batch_of_token(const oracle_problem *p, int64_t tok)
{
    for (int b = 0; b < p->B; ++b)
        if (tok >= p->cu_q[b] && tok < p->cu_q[b + 1])
            return b;
    return -1;
}

/* One output row.  s is scratch of length >= Lk. */
static void one_row(const oracle_problem *p, int b, int64_t tok, int h, double *s,
                    double *o_row, double *lse_out)
{
    const int G = p->Hq / p->Hkv;
#if ORACLE_MUTANT == 2
    const int g = h % p->Hkv; /* wrong GQA head map */
#else
    const int g = h / G;
#endif
    const int64_t Lq = p->cu_q[b + 1] - p->cu_q[b];
    const int64_t Lk = p->cu_k[b + 1] - p->cu_k[b];
    const int64_t i = tok - p->cu_q[b];
#if ORACLE_MUTANT == 3
    const int64_t delta = 0; /* top-left causal alignment */
#else
    const int64_t delta = Lk - Lq;
#endif
    const double dqs = p->dq[b * p->Hkv + g];
    const double dks = p->dk[b * p->Hkv + g];
    const double dvs = p->dv[b * p->Hkv + g];
#if ORACLE_MUTANT == 4
    const double scale = p->softmax_scale * dqs; /* dropped k descale */
#else
    const double scale = p->softmax_scale * dqs * dks;
#endif

    int64_t hi = Lk - 1, lo = 0;
    if (p->causal && i + delta < hi)
        hi = i + delta;
#if ORACLE_MUTANT == 8
    if (p->window_left >= 0 && i + delta - p->window_left + 1 > lo)
        lo = i + delta - p->window_left + 1; /* window one key short */
#else
    if (p->window_left >= 0 && i + delta - p->window_left > lo)
        lo = i + delta - p->window_left;
#endif

    const uint8_t *qrow = p->q + (tok * p->Hq + h) * (int64_t)p->D;
    double m = -INFINITY;
    for (int64_t j = lo; j <= hi; ++j) {
        const uint8_t *krow = key_row(p, p->k, p->D, b, g, j);
        double acc = 0.0;
        for (int t = 0; t < p->D; ++t) {
#if ORACLE_MUTANT == 5
            acc += oracle_e4m3_decode(qrow[t]) * oracle_e4m3_decode(krow[p->D - 1 - t]);
#else
            acc += oracle_e4m3_decode(qrow[t]) * oracle_e4m3_decode(krow[t]);
#endif
        }
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    const int has_sink = p->sink != NULL;
    const double sk = has_sink ? p->sink[h] : -INFINITY;
    if (sk > m)
        m = sk;

    for (int c = 0; c < p->DV; ++c)
        o_row[c] = 0.0;
    if (m == -INFINITY) { /* nothing visible and no sink */
        *lse_out = -INFINITY;
        return;
    }
    double Z = 0.0;
    for (int64_t j = lo; j <= hi; ++j) {
        double w = exp(s[j] - m);
        Z += w;
        const uint8_t *vrow = key_row(p, p->v, p->DV, b, g, j);
        for (int c = 0; c < p->DV; ++c) {
#if ORACLE_MUTANT == 10
            /* O accumulated in fp32 with every add truncated toward zero: a reduced-precision
               accumulator whose rounding loss grows with the key count */
            o_row[c] = truncf_add((float)o_row[c], (float)(w * oracle_e4m3_decode(vrow[c])));
#else
            o_row[c] += w * oracle_e4m3_decode(vrow[c]);
#endif
        }
    }
#if ORACLE_MUTANT == 6
    (void)sk; /* sink dropped from the denominator */
#else
    if (has_sink)
        Z += exp(sk - m);
#endif
    for (int c = 0; c < p->DV; ++c) {
#if ORACLE_MUTANT == 7
        o_row[c] = o_row[c] / Z; /* v descale dropped */
#else
        o_row[c] = dvs * o_row[c] / Z;
#endif
    }
    (void)dvs;
#if ORACLE_MUTANT == 9
    *lse_out = log(Z); /* max shift not added back */
#else
    *lse_out = m + log(Z);
#endif
}

/*
 * n_rows < 0 : computes O [total_q][Hq][DV] and LSE [total_q][Hq] (row-major, fp64)
 *              for every (token, head).
 * n_rows >= 0: computes only the listed (token, head) pairs, compactly:
 *              O [n_rows][DV], LSE [n_rows].
 * Returns 0, or -1 on a malformed problem / allocation failure.
 */
int oracle_attention(const oracle_problem *p, double *o, double *lse)
{
    if (!p || p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Hq % p->Hkv != 0)
        return -1;
    int64_t max_lk = 0;
    for (int b = 0; b < p->B; ++b) {
        int64_t lk = p->cu_k[b + 1] - p->cu_k[b];
        if (lk < 0 || p->cu_q[b + 1] < p->cu_q[b])
            return -1;
        if (lk > max_lk)
            max_lk = lk;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
    if (!s)
        return -1;
    const int64_t total_q = p->cu_q[p->B];
    if (p->n_rows < 0) {
        for (int64_t tok = 0; tok < total_q; ++tok) {
            int b = batch_of_token(p, tok);
            for (int h = 0; h < p->Hq; ++h)
                one_row(p, b, tok, h, s, o + (tok * p->Hq + h) * (int64_t)p->DV,
                        lse + tok * p->Hq + h);
        }
    } else {
        for (int64_t r = 0; r < p->n_rows; ++r) {
            int64_t tok = p->rows_tok[r];
            int h = p->rows_head[r];
            int b = batch_of_token(p, tok);
            if (b < 0 || h < 0 || h >= p->Hq) {
                free(s);
                return -1;
            }
            one_row(p, b, tok, h, s, o + r * (int64_t)p->DV, lse + r);
        }
    }
    free(s);
    return 0;
}
