/*
 * Float64 CPU oracle for speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the verification hot path computes.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant with the CUDA library: the
 * dtype codes below are this file's own.
 *
 * Two operations, each written as its plain definition:
 *
 *  1. Multi-query causal attention of k draft-token queries over a paged
 *     KV cache ("Decoding Speculative Decoding from First Principles",
 *     sections "Parallelizing method 2: sequence parallel" and "Speculating
 *     to get sequence parallelism during decode": the target runs the
 *     drafted tokens through one prefill-style pass, so each draft query
 *     attends to the whole cached context plus the drafts up to and
 *     including its own position).  Optional INT8 cache: the dequantiser is
 *     the inverse of "Algorithm 2 KV-Cache Compression" on the CXL-SpecKV
 *     page (s = max|X|/127, c = round(X/s), so X ~ c*s), at per-(token,
 *     kv-head) granularity with an fp16 scale.
 *
 *  2. Greedy longest-prefix acceptance ("Decoding Speculative Decoding from
 *     First Principles", section "Speculating to get sequence parallelism
 *     during decode"): the target's prediction at every drafted position is
 *     its argmax; drafts are kept up to the first disagreement, where the
 *     target's own token is emitted; if every draft agrees, the prediction
 *     after the last draft is the extra ("bonus") token.  One pass therefore
 *     yields between 1 and k+1 tokens.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   - ctx_lens excludes the drafts; query i of sequence b sits at position
 *     ctx_b + i and sees keys 0 .. ctx_b + i inclusive.
 *   - acceptance takes k+1 logits rows per sequence: row i predicts draft
 *     i, row k predicts the bonus token.
 *   - argmax ties resolve to the lowest vocabulary index; values compare as
 *     the float64 widening of the stored bits (so -0 == +0).
 *   - lse is the natural-log log-sum-exp of the scaled scores.
 *
 * Layouts (row-major, element strides implied):
 *   q            [B, k, Hq, D]          f32 | bf16 | f16
 *   k/v cache    [NP, Hkv, P, D]        f32 | bf16 | f16 | i8
 *   k/v scale    [NP, Hkv, P]           f16 bits (only with an i8 cache)
 *   block_table  [B, max_pages]         int32 physical page ids
 *   ctx_lens     [B]                    int32
 *   logits       [B, k+1, V]            f32 | bf16 | f16
 *   draft        [B, k]                 int32
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* This file's own element-type codes. */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_I8 = 3 };

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);            /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1+frac/1024)*2^(e-15) */
    return sign ? -mag : mag;
}

static double load_f64(const void *base, int dtype, int64_t idx) {
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[idx];
    case ORC_BF16: return bf16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_F16: return f16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_I8: return (double)((const int8_t *)base)[idx];
    default: return NAN;
    }
}

double oracle_bf16_to_f64(uint16_t bits) { return bf16_to_f64(bits); }
double oracle_f16_to_f64(uint16_t bits) { return f16_to_f64(bits); }

typedef struct {
    const void *q; int q_dtype;
    const void *k_cache; const void *v_cache; int kv_dtype;
    const uint16_t *k_scale; const uint16_t *v_scale;
    const int32_t *block_table; const int32_t *ctx_lens;
    int B, num_draft, Hq, Hkv, D, P, num_pages, max_pages;
    double scale;
} attn_args;

/* Dequantised element d of cached row (sequence b, logical key j, kv-head g). */
static double cache_elem(const attn_args *a, const void *cache, const uint16_t *scale,
                         int b, int64_t j, int g, int d, int *bad) {
    int64_t logical_page = j / a->P;
    int slot = (int)(j % a->P);
    if (logical_page >= a->max_pages) { *bad = 1; return 0.0; }
    int32_t page = a->block_table[(int64_t)b * a->max_pages + logical_page];
    if (page < 0 || page >= a->num_pages) { *bad = 1; return 0.0; }
    int64_t row = ((int64_t)page * a->Hkv + g) * a->P + slot;
    double x = load_f64(cache, a->kv_dtype, row * a->D + d);
    if (a->kv_dtype == ORC_I8) x *= f16_to_f64(scale[row]);  /* X = c * s */
    return x;
}

/*
 * One output row: sequence b, draft position i, query head h.
 * out_row[D] receives sum_j softmax(s)_j * V_j and *lse_out the natural-log
 * log-sum-exp of s.  Returns 0, or -1 on an out-of-range page reference.
 */
static int attn_row(const attn_args *a, int b, int i, int h, double *out_row, double *lse_out) {
    int G = a->Hq / a->Hkv;
    int g = h / G;                                  /* GQA: kv-head serving q-head h */
    int64_t n_keys = (int64_t)a->ctx_lens[b] + i + 1; /* causal: keys 0 .. ctx_b + i */
    int bad = 0;
    const int64_t q_off = (((int64_t)b * a->num_draft + i) * a->Hq + h) * a->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    if (!s) return -2;

    /* scores s_j = scale * <q, K_j> */
    for (int64_t j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int d = 0; d < a->D; ++d)
            dot += load_f64(a->q, a->q_dtype, q_off + d) *
                   cache_elem(a, a->k_cache, a->k_scale, b, j, g, d, &bad);
        s[j] = a->scale * dot;
    }
    if (bad) { free(s); return -1; }

    /* two-pass softmax: max, then log-sum-exp */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) sum += exp(s[j] - m);
    double lse = m + log(sum);

    /* out = sum_j exp(s_j - lse) * V_j */
    for (int d = 0; d < a->D; ++d) out_row[d] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        double p = exp(s[j] - lse);
        for (int d = 0; d < a->D; ++d)
            out_row[d] += p * cache_elem(a, a->v_cache, a->v_scale, b, j, g, d, &bad);
    }
    free(s);
    *lse_out = lse;
    return bad ? -1 : 0;
}

static int check_shape(const attn_args *a) {
    if (a->B < 0 || a->num_draft < 1 || a->Hq < 1 || a->Hkv < 1 || a->D < 1 || a->P < 1) return -1;
    if (a->Hq % a->Hkv) return -1;
    if (a->kv_dtype == ORC_I8 && (!a->k_scale || !a->v_scale)) return -1;
    return 0;
}

#define ATTN_ARGS_INIT                                                              \
    attn_args a = {q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,        \
                   block_table, ctx_lens, B, num_draft, Hq, Hkv, D, P, num_pages,   \
                   max_pages, scale}

/* Full attention: out [B, k, Hq, D] and lse [B, k, Hq], both float64. */
int oracle_verify_attn(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                       int kv_dtype, const uint16_t *k_scale, const uint16_t *v_scale,
                       const int32_t *block_table, const int32_t *ctx_lens, int B, int num_draft,
                       int Hq, int Hkv, int D, int P, int num_pages, int max_pages, double scale,
                       double *out, double *lse) {
    ATTN_ARGS_INIT;
    if (check_shape(&a)) return -1;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < num_draft; ++i)
            for (int h = 0; h < Hq; ++h) {
                int64_t r = ((int64_t)b * num_draft + i) * Hq + h;
                int rc = attn_row(&a, b, i, h, out + r * D, lse + r);
                if (rc) return rc;
            }
    return 0;
}

/* Selected rows only: rows[3*n] = (b, i, h); out [n, D], lse [n]. */
int oracle_attn_rows(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                     int kv_dtype, const uint16_t *k_scale, const uint16_t *v_scale,
                     const int32_t *block_table, const int32_t *ctx_lens, int B, int num_draft,
                     int Hq, int Hkv, int D, int P, int num_pages, int max_pages, double scale,
                     const int32_t *rows, int n_rows, double *out, double *lse) {
    ATTN_ARGS_INIT;
    if (check_shape(&a)) return -1;
    for (int r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], i = rows[3 * r + 1], h = rows[3 * r + 2];
        if (b < 0 || b >= B || i < 0 || i >= num_draft || h < 0 || h >= Hq) return -1;
        int rc = attn_row(&a, b, i, h, out + (int64_t)r * D, lse + r);
        if (rc) return rc;
    }
    return 0;
}

/* First index of the maximum of one row, comparing float64 widenings. */
static int32_t row_argmax(const void *logits, int dtype, int64_t row_off, int64_t V) {
    int32_t best = 0;
    double best_v = load_f64(logits, dtype, row_off);
    for (int64_t v = 1; v < V; ++v) {
        double x = load_f64(logits, dtype, row_off + v);
        if (x > best_v) { best_v = x; best = (int32_t)v; }
    }
    return best;
}

/*
 * Greedy acceptance.  logits [B, k+1, V]; draft [B, k].
 * accepted_len[b] = number of leading drafts equal to the target argmax;
 * next_token[b]   = target argmax at position accepted_len[b] (the
 *                   correction token, or the bonus token when all k agree).
 * argmax_rows [B, k+1] (optional) receives every row's argmax.
 */
int oracle_accept_greedy(const void *logits, int dtype, const int32_t *draft, int B,
                         int num_draft, int64_t V, int32_t *accepted_len, int32_t *next_token,
                         int32_t *argmax_rows) {
    if (B < 0 || num_draft < 1 || V < 1) return -1;
    int32_t *a = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_draft + 1));
    if (!a) return -2;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i <= num_draft; ++i)
            a[i] = row_argmax(logits, dtype, ((int64_t)b * (num_draft + 1) + i) * V, V);
        int n = 0;
        while (n < num_draft && draft[(int64_t)b * num_draft + n] == a[n]) ++n;
        accepted_len[b] = n;
        next_token[b] = a[n];
        if (argmax_rows)
            for (int i = 0; i <= num_draft; ++i) argmax_rows[(int64_t)b * (num_draft + 1) + i] = a[i];
    }
    free(a);
    return 0;
}
