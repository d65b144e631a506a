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
    const uint64_t *tree_mask; /* [B, k] or NULL (causal chain) */
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
/*
 * Keys visible to draft query i of sequence b: the whole cached context
 * 0 .. ctx_b - 1, then draft position t (key ctx_b + t) when the query may
 * see it -- t <= i for the causal chain, or bit t of tree_mask[b][i] for a
 * tree of drafts (each node sees its ancestors and itself; SpecInfer-style
 * tree verification, "Decoding Speculative Decoding from First Principles",
 * section "Advances in speculators").
 */
static int64_t visible_keys(const attn_args *a, int b, int i, int64_t *keys) {
    const int64_t ctx = a->ctx_lens[b];
    int64_t n = 0;
    for (int64_t j = 0; j < ctx; ++j) keys[n++] = j;
    for (int t = 0; t < a->num_draft; ++t) {
        const int vis = a->tree_mask ? (int)((a->tree_mask[(int64_t)b * a->num_draft + i] >> t) & 1u)
                                     : t <= i;
        if (vis) keys[n++] = ctx + t;
    }
    return n;
}

static int attn_row(const attn_args *a, int b, int i, int h, double *out_row, double *lse_out) {
    int G = a->Hq / a->Hkv;
    int g = h / G;                                  /* GQA: kv-head serving q-head h */
    int bad = 0;
    const int64_t q_off = (((int64_t)b * a->num_draft + i) * a->Hq + h) * a->D;
    const int64_t cap = (int64_t)a->ctx_lens[b] + a->num_draft;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    if (!s || !keys) { free(s); free(keys); return -2; }
    const int64_t n_keys = visible_keys(a, b, i, keys);

    /* scores s_j = scale * <q, K_j> over the visible keys */
    for (int64_t jj = 0; jj < n_keys; ++jj) {
        double dot = 0.0;
        for (int d = 0; d < a->D; ++d)
            dot += load_f64(a->q, a->q_dtype, q_off + d) *
                   cache_elem(a, a->k_cache, a->k_scale, b, keys[jj], g, d, &bad);
        s[jj] = a->scale * dot;
    }
    if (bad) { free(s); free(keys); return -1; }

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
            out_row[d] += p * cache_elem(a, a->v_cache, a->v_scale, b, keys[j], g, d, &bad);
    }
    free(s);
    free(keys);
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
                   max_pages, scale, NULL}

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

/*
 * 3. Rejection-sampling acceptance ("Decoding Speculative Decoding from First
 *    Principles", section "How does this drafter maintain the same
 *    distribution of the target?").  p is the target's next-token
 *    distribution and q the drafter's, each softmax(logits / T).  At every
 *    drafted position the draft x is kept with probability min(1, p(x)/q(x))
 *    (always when p(x) >= q(x)); at the first rejection a token is drawn from
 *    the residual max(p - q, 0), renormalised; when all k drafts are kept the
 *    bonus token is drawn from p at position k.  The emitted tokens then
 *    follow p exactly (the section's "Proving the same distribution").
 *
 *    Random draws.  Every draw comes from the counter-based generator
 *    SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *    generators", 2014): the n-th output for seed s is the SplitMix64 mix of
 *    s + (n + 1) * 0x9E3779B97F4A7C15.  Draw n = ((2 b + kind) << 32) | j:
 *      kind 0, j = position i: the acceptance uniform u in [0, 1) (24 bits);
 *      kind 1, j = token x:    the Gumbel noise g = -ln(-ln u'), u' in (0, 1).
 *    A draw from a distribution w over the vocabulary is the Gumbel-max
 *    choice argmax_x ln w(x) + g(x) (lowest index on ties), which picks x
 *    with probability w(x) / sum w.
 *
 *    target [B, k+1, V], draft_logits [B, k, V] (same dtype), draft [B, k].
 *    Optional diagnostics: ratio / unif [B, k] receive p(x)/q(x) and u at
 *    every position up to the first rejection (NaN after it); key_gap [B]
 *    the gap between the best and second-best Gumbel keys of the draw.
 */
static uint64_t sm64_at(uint64_t seed, uint64_t n) {
    uint64_t z = seed + (n + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* The n-th SplitMix64 output (exported for the generator's known-answer pin). */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t n) { return sm64_at(seed, n); }

static uint64_t draw_index(int b, int kind, int64_t j) {
    return ((uint64_t)(2 * (uint64_t)b + (uint64_t)kind) << 32) | (uint64_t)j;
}

/* 24-bit uniform in [0, 1) and in (0, 1). */
static double unif_co(uint64_t z) { return (double)(z >> 40) * 0x1p-24; }
static double unif_oo(uint64_t z) { return (double)((z >> 41) * 2 + 1) * 0x1p-24; }

double oracle_accept_uniform(uint64_t seed, int b, int i) {
    return unif_co(sm64_at(seed, draw_index(b, 0, i)));
}

double oracle_gumbel(uint64_t seed, int b, int64_t x) {
    return -log(-log(unif_oo(sm64_at(seed, draw_index(b, 1, x)))));
}

/* ln sum_x exp(row[x] / T) */
static double row_lse(const void *logits, int dtype, int64_t off, int64_t V, double T) {
    double m = -INFINITY;
    for (int64_t x = 0; x < V; ++x) {
        double l = load_f64(logits, dtype, off + x) / T;
        if (l > m) m = l;
    }
    double s = 0.0;
    for (int64_t x = 0; x < V; ++x) s += exp(load_f64(logits, dtype, off + x) / T - m);
    return m + log(s);
}

int oracle_accept_rejection(const void *target, const void *draft_logits, int dtype,
                            const int32_t *draft, int B, int num_draft, int64_t V,
                            double temperature, uint64_t seed, int32_t *accepted_len,
                            int32_t *next_token, double *ratio, double *unif, double *key_gap) {
    if (B < 0 || num_draft < 1 || V < 1 || !(temperature > 0.0)) return -1;
    const double T = temperature;
    const int k = num_draft;
    for (int b = 0; b < B; ++b) {
        int n = k;
        double lse_p = 0.0, lse_q = 0.0;
        for (int i = 0; i < k; ++i) {
            const int32_t x = draft[(int64_t)b * k + i];
            if (x < 0 || x >= V) return -1;
            const int64_t po = ((int64_t)b * (k + 1) + i) * V, qo = ((int64_t)b * k + i) * V;
            lse_p = row_lse(target, dtype, po, V, T);
            lse_q = row_lse(draft_logits, dtype, qo, V, T);
            const double lp = load_f64(target, dtype, po + x) / T - lse_p;
            const double lq = load_f64(draft_logits, dtype, qo + x) / T - lse_q;
            const double r = exp(lp - lq);  /* p(x) / q(x) */
            const double u = oracle_accept_uniform(seed, b, i);
            if (ratio) ratio[(int64_t)b * k + i] = r;
            if (unif) unif[(int64_t)b * k + i] = u;
            if (!(u < r)) { n = i; break; }
        }
        if (ratio)
            for (int i = n + 1; i < k; ++i) ratio[(int64_t)b * k + i] = NAN;
        if (unif)
            for (int i = n + 1; i < k; ++i) unif[(int64_t)b * k + i] = NAN;
        /* Gumbel-max draw: from p at position k (bonus) or from the residual at n */
        double best = -INFINITY, second = -INFINITY;
        int32_t arg = -1;
        const int64_t po = ((int64_t)b * (k + 1) + n) * V, qo = ((int64_t)b * k + n) * V;
        for (int64_t x = 0; x < V; ++x) {
            double lw;
            if (n == k) {
                lw = load_f64(target, dtype, po + x) / T;  /* ln p(x) up to a constant */
            } else {
                const double p = exp(load_f64(target, dtype, po + x) / T - lse_p);
                const double q = exp(load_f64(draft_logits, dtype, qo + x) / T - lse_q);
                const double w = p - q;
                lw = w > 0.0 ? log(w) : -INFINITY;
            }
            if (lw == -INFINITY) continue;
            const double key = lw + oracle_gumbel(seed, b, x);
            if (key > best) { second = best; best = key; arg = (int32_t)x; }
            else if (key > second) second = key;
        }
        if (arg < 0) return -3; /* an empty residual cannot follow a rejection */
        accepted_len[b] = n;
        next_token[b] = arg;
        if (key_gap) key_gap[b] = best - second;
    }
    return 0;
}

/*
 * 4. Writing the drafts' K/V rows into the paged cache, and the commit.
 *
 *    The drafted positions ctx_b .. ctx_b + n - 1 of sequence b get the new
 *    rows k_new / v_new [B, n, Hkv, D] (f32 or bf16) at page
 *    block_table[b][pos / P], slot pos % P.  An f32 or bf16 cache stores the
 *    value (bf16 rounded to nearest even); an INT8 cache stores the
 *    quantised row of CXL-SpecKV's "Algorithm 2 KV-Cache Compression" (steps
 *    "Scaling" and "Quantization"), per (token, kv-head) row:
 *      s = fp16(max_d |x_d| / 127), c_d = clamp(rint(x_d / s), -127, 127),
 *      and c = 0 when s = 0.
 *    The quantiser decides integers, so it takes the kernel's precision:
 *    every step in fp32 (IEEE division, round half to even), the scale
 *    rounded to binary16 by round-to-nearest-even.
 *
 *    The commit is the KVMU's Accept pointer move (HeteroReason, KV Cache
 *    Management Unit): the validated length of sequence b grows by its
 *    accepted drafts (plus `extra`, 1 when the emitted token's row is counted
 *    too); rejected drafts are not advanced over, so the next step's append
 *    overwrites them (the Rollback).
 */

/* float -> IEEE binary16 bits, round to nearest even; overflow -> inf. */
static uint16_t f32_to_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    const double v = fabs((double)f);
    if (v != v) return sign | 0x7e00u;
    if (v >= 65520.0) return sign | 0x7c00u;          /* beyond the largest finite half */
    if (v < ldexp(1.0, -14)) {                        /* subnormal range: multiples of 2^-24 */
        const double r = rint(v * ldexp(1.0, 24));     /* exact scaling, round half even */
        return sign | (uint16_t)r;                     /* r == 1024 is the smallest normal */
    }
    int e2;
    frexp(v, &e2);                                    /* v in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    double r = rint(ldexp(v, 10 - E));                /* in [1024, 2048] */
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E + 15 >= 31) return sign | 0x7c00u;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/* float -> bfloat16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    return (uint16_t)((x + 0x7fffu + ((x >> 16) & 1u)) >> 16);
}

static void quantize_row(const void *src, int src_dtype, int64_t off, int D, int8_t *codes,
                         uint16_t *scale_bits) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float v = fabsf((float)load_f64(src, src_dtype, off + d));
        if (v > amax) amax = v;
    }
    const float sf = amax / 127.0f;
    const uint16_t sb = f32_to_f16_bits(sf);
    const float s = (float)f16_to_f64(sb);
    for (int d = 0; d < D; ++d) {
        float c = 0.0f;
        if (s > 0.0f) {
            const float q = (float)load_f64(src, src_dtype, off + d) / s;
            c = rintf(q);
            if (c > 127.0f) c = 127.0f;
            if (c < -127.0f) c = -127.0f;
        }
        codes[d] = (int8_t)c;
    }
    *scale_bits = sb;
}

/* Rows [n, D] of src -> codes [n, D] int8 and scale bits [n] (fp16). */
int oracle_quantize_rows(const void *src, int src_dtype, int64_t n, int D, int8_t *codes,
                         uint16_t *scale_bits) {
    if (n < 0 || D < 1) return -1;
    for (int64_t r = 0; r < n; ++r)
        quantize_row(src, src_dtype, r * D, D, codes + r * D, scale_bits + r);
    return 0;
}

int oracle_kv_append(const void *k_new, const void *v_new, int src_dtype, void *k_cache,
                     void *v_cache, uint16_t *k_scale, uint16_t *v_scale, int cache_dtype,
                     const int32_t *block_table, const int32_t *ctx_lens, int B, int n_new,
                     int Hkv, int D, int P, int num_pages, int max_pages) {
    if (B < 0 || n_new < 1 || Hkv < 1 || D < 1 || P < 1) return -1;
    if (src_dtype != ORC_F32 && src_dtype != ORC_BF16) return -1;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < n_new; ++t) {
            const int64_t pos = (int64_t)ctx_lens[b] + t;
            if (pos < 0 || pos / P >= max_pages) return -1;
            const int32_t page = block_table[(int64_t)b * max_pages + pos / P];
            if (page < 0 || page >= num_pages) return -1;
            for (int g = 0; g < Hkv; ++g) {
                const int64_t srow = (((int64_t)b * n_new + t) * Hkv + g) * D;
                const int64_t crow = (((int64_t)page * Hkv + g) * P + pos % P);
                for (int tensor = 0; tensor < 2; ++tensor) {
                    const void *src = tensor ? v_new : k_new;
                    void *cache = tensor ? v_cache : k_cache;
                    if (cache_dtype == ORC_I8) {
                        uint16_t *sc = tensor ? v_scale : k_scale;
                        quantize_row(src, src_dtype, srow, D, (int8_t *)cache + crow * D, sc + crow);
                    } else {
                        for (int d = 0; d < D; ++d) {
                            const float v = (float)load_f64(src, src_dtype, srow + d);
                            if (cache_dtype == ORC_F32)
                                ((float *)cache)[crow * D + d] = v;
                            else if (cache_dtype == ORC_BF16)
                                ((uint16_t *)cache)[crow * D + d] = f32_to_bf16_bits(v);
                            else
                                return -1;
                        }
                    }
                }
            }
        }
    return 0;
}

int oracle_commit(int32_t *ctx_lens, const int32_t *accepted_len, int B, int extra) {
    for (int b = 0; b < B; ++b) ctx_lens[b] += accepted_len[b] + extra;
    return 0;
}

/* Tree attention: as oracle_verify_attn, query i of sequence b seeing the
 * context and the drafts set in tree_mask[b][i] (see visible_keys). */
int oracle_verify_attn_tree(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                            int kv_dtype, const uint16_t *k_scale, const uint16_t *v_scale,
                            const int32_t *block_table, const int32_t *ctx_lens, int B,
                            int num_draft, int Hq, int Hkv, int D, int P, int num_pages,
                            int max_pages, double scale, const uint64_t *tree_mask, double *out,
                            double *lse) {
    ATTN_ARGS_INIT;
    a.tree_mask = tree_mask;
    if (check_shape(&a) || num_draft > 64) return -1;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < num_draft; ++i)
            for (int h = 0; h < Hq; ++h) {
                const int64_t r = ((int64_t)b * num_draft + i) * Hq + h;
                int rc = attn_row(&a, b, i, h, out + r * D, lse + r);
                if (rc) return rc;
            }
    return 0;
}

/*
 * 5. Greedy acceptance over a tree of drafts (SpecInfer / EAGLE-style token
 *    trees, "Advances in speculators"): node i carries token draft[b][i]
 *    and parent parent[b][i] in [-1, i) (-1: a child of the last committed
 *    token).  logits row 0 is the target's prediction at the root, row i+1
 *    its prediction after node i.  From the root, the walk keeps the child
 *    whose token equals the target's argmax at the current node (the lowest
 *    index if several do), and stops when none does; accepted_len is the
 *    path length, next_token the argmax after the last kept node, path
 *    [B, k] the kept nodes in order (-1 after the end).  A chain
 *    (parent[i] = i - 1) is the greedy rule of section 2.
 */
int oracle_accept_tree(const void *logits, int dtype, const int32_t *draft, const int32_t *parent,
                       int B, int num_draft, int64_t V, int32_t *accepted_len,
                       int32_t *next_token, int32_t *path) {
    if (B < 0 || num_draft < 1 || V < 1) return -1;
    const int k = num_draft;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < k; ++i) {
            const int32_t p = parent[(int64_t)b * k + i];
            if (p < -1 || p >= i) return -1;
        }
        int cur = -1, n = 0;
        for (int i = 0; i < k; ++i) path[(int64_t)b * k + i] = -1;
        for (;;) {
            const int32_t a = row_argmax(logits, dtype, ((int64_t)b * (k + 1) + cur + 1) * V, V);
            int next = -1;
            for (int c = 0; c < k && next < 0; ++c)
                if (parent[(int64_t)b * k + c] == cur && draft[(int64_t)b * k + c] == a) next = c;
            if (next < 0) {
                accepted_len[b] = n;
                next_token[b] = a;
                break;
            }
            path[(int64_t)b * k + n++] = next;
            cur = next;
        }
    }
    return 0;
}

/* ---- Delta + run-length page codec (CXL-SpecKV: observation (5), "spatial
 * correlation of attention heads ... delta coding delta_i = x_i - x_(i-1)",
 * and "Algorithm 2 KV-Cache Compression", whose output is (s, D_RLE(c)); the
 * ablation credits INT8 2.00x, delta +36 %, RLE +18 %).  The page gives the
 * two steps, not a byte format; this one is the plainest that is lossless:
 *   - a block is the P x D INT8 codes of one (page, kv-head), row-major;
 *   - delta along the head dimension inside each row, in arithmetic modulo
 *     256 on the code bytes: e[r][0] = c[r][0], e[r][d] = c[r][d] - c[r][d-1];
 *   - the block's stream e (row-major) becomes maximal runs of equal bytes,
 *     each run stored as the byte pair (length 1..255, value); a run longer
 *     than 255 continues in the next pair.
 * The fp16 scales are not coded. */
int oracle_codec_encode(const int8_t *codes, int64_t nblk, int P, int D, uint8_t *pairs,
                        int32_t *npairs) {
    const int64_t n = (int64_t)P * D;
    uint8_t *e = (uint8_t *)malloc((size_t)n);
    if (!e) return -1;
    for (int64_t blk = 0; blk < nblk; ++blk) {
        const uint8_t *c = (const uint8_t *)codes + blk * n;
        for (int r = 0; r < P; ++r)
            for (int d = 0; d < D; ++d) {
                const uint8_t prev = d ? c[(int64_t)r * D + d - 1] : 0;
                e[(int64_t)r * D + d] = (uint8_t)(c[(int64_t)r * D + d] - prev);
            }
        uint8_t *out = pairs + blk * 2 * n;
        int64_t np = 0;
        for (int64_t i = 0; i < n;) {
            const uint8_t v = e[i];
            int len = 1;
            while (i + len < n && e[i + len] == v && len < 255) ++len;
            out[2 * np] = (uint8_t)len;
            out[2 * np + 1] = v;
            ++np;
            i += len;
        }
        npairs[blk] = (int32_t)np;
    }
    free(e);
    return 0;
}

/* Inverse: expand the pairs, then sum each row's deltas modulo 256.  Returns
 * -1 for a block whose pair count is outside [0, P*D] or whose lengths do
 * not sum to P*D (nothing past the block is written). */
int oracle_codec_decode(const uint8_t *pairs, const int32_t *npairs, int64_t nblk, int P, int D,
                        int8_t *codes) {
    const int64_t n = (int64_t)P * D;
    int bad = 0;
    for (int64_t blk = 0; blk < nblk; ++blk) {
        uint8_t *c = (uint8_t *)codes + blk * n;
        const uint8_t *in = pairs + blk * 2 * n;
        const int64_t np = npairs[blk];
        int64_t pos = 0;
        if (np < 0 || np > n) { bad = 1; continue; }
        for (int64_t j = 0; j < np; ++j) {
            const int len = in[2 * j];
            for (int t = 0; t < len && pos < n; ++t) c[pos++] = in[2 * j + 1];
            if (len == 0) bad = 1;
        }
        if (pos != n) { bad = 1; continue; }
        for (int r = 0; r < P; ++r) {
            uint8_t acc = 0;
            for (int d = 0; d < D; ++d) {
                acc = (uint8_t)(acc + c[(int64_t)r * D + d]);
                c[(int64_t)r * D + d] = acc;
            }
        }
    }
    return bad ? -1 : 0;
}
