/*
 * dsa_oracle.c -- plain, slow, single-threaded CPU definition of one DeepSeek
 * Sparse Attention (DSA) layer, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library, and it never reads anything
 * the CUDA library produced.
 *
 * Source passages (page title, then section):
 *   "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
 *     section "Model and bottleneck": DSA reads about 2048 keys per query; its
 *     indexer scores one pool per 4 tokens for every query.
 *   same page, section "1. DSA truly sparse": the Flash variant uses no
 *     positional encoding (NoPE), selects 2051 rather than 2048 keys, scores
 *     the indexer in query chunks, and passes selected pool indices as int32.
 * The pages print no formula.  The readings taken here, each the plainest one
 * the passages support:
 *   - pool key: kpool[p] = k_I[4p] + k_I[4p+1] + k_I[4p+2] + k_I[4p+3], added
 *     in that order in fp32 and, for bf16 layers, rounded once to bf16 (round
 *     to nearest, ties to even).  This is the value the layer stores.
 *   - eligibility: pool p is visible to query t iff all its tokens are <= t,
 *     i.e. p < elig(t) = floor((t+1)/4).
 *   - score: s[t,p] = sum_h w[t,h] * max(0, q_I[t,h,:] . kpool[p,:]).
 *   - selection: the first min(k, elig(t)) pools under the order
 *     (score descending, pool index ascending); reported in ascending pool
 *     order, padded with -1.  -0 and +0 compare equal.
 *   - key set: the tokens of the selected pools, plus the query's own partial
 *     pool 4*floor(t/4) .. t when t mod 4 != 3 (at most 4k+3 keys: 2051 at
 *     k=512).  When t mod 4 == 3 the own pool is complete and competes in
 *     the selection like any other pool.
 *   - attention: one shared K/V head (no positional encoding), softmax with
 *     scale `scale`, O = softmax(S) V and LSE = log sum exp S (natural log).
 *   - backward: the analytic gradients of that attention; the selection is
 *     piecewise constant, so the indexer inputs receive no gradient.
 * Every input array holds the exact values of the layer's typed inputs
 * (bf16 values are exact in fp32); all arithmetic after the pool key is in
 * double.  There is no blocking, fusion or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_INDEX 1   /* an idx entry names a pool outside 0..elig(t)-1 */
#define ORACLE_NO_MEMORY 2

static int64_t elig(int64_t t) { return (t + 1) / 4; }

/* fp32 -> nearest bf16 value (ties to even), returned as fp32.  Written from
 * the definition: keep the top 16 bits of the fp32 pattern after adding half
 * an ulp of the kept part, plus one when the kept part is odd (the tie goes
 * to the even neighbour).  NaN stays NaN. */
float oracle_round_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0) {
        u |= 0x00400000u;
        u &= 0xffff0000u;
    } else {
        uint32_t keep_lsb = (u >> 16) & 1u;
        u += 0x7fffu + keep_lsb;
        u &= 0xffff0000u;
    }
    float y;
    memcpy(&y, &u, 4);
    return y;
}

/* Pool keys (page 1, "Model and bottleneck": one pool per 4 tokens).
 * k_I: [L, di]; kpool: [L/4, di]. */
void oracle_pool_keys(int64_t L, int32_t di, int32_t round_to_bf16,
                      const float *k_I, float *kpool)
{
    int64_t P = L / 4;
    for (int64_t p = 0; p < P; ++p) {
        for (int32_t i = 0; i < di; ++i) {
            float s = k_I[(4 * p + 0) * di + i];
            s = s + k_I[(4 * p + 1) * di + i];
            s = s + k_I[(4 * p + 2) * di + i];
            s = s + k_I[(4 * p + 3) * di + i];
            kpool[p * di + i] = round_to_bf16 ? oracle_round_bf16(s) : s;
        }
    }
}

/* Gated pool keys: the same pools, each token's key weighted by a per-token
 * gate before the sum (page 1, "3. Context parallelism (CP)", names "k-pool
 * gate scores" aligned with the keys and defines nothing more).  Reading:
 * kpool[p] = sum_{j<4} gate[4p+j] * k_I[4p+j], accumulated in fp32 in token
 * order with one fused multiply-add per token (acc = fma(g, k, acc) from
 * acc = 0), then rounded once to the layer dtype.  With every gate 1 it is
 * oracle_pool_keys exactly.  k_I: [L, di]; gate: [L]; kpool: [L/4, di]. */
void oracle_pool_keys_gated(int64_t L, int32_t di, int32_t round_to_bf16,
                            const float *k_I, const float *gate, float *kpool)
{
    int64_t P = L / 4;
    for (int64_t p = 0; p < P; ++p) {
        for (int32_t i = 0; i < di; ++i) {
            float s = 0.0f;
            for (int j = 0; j < 4; ++j)
                s = fmaf(gate[4 * p + j], k_I[(4 * p + j) * di + i], s);
            kpool[p * di + i] = round_to_bf16 ? oracle_round_bf16(s) : s;
        }
    }
}

/* Indexer scores for the listed query rows (page 1, "Model and bottleneck":
 * every query scores every pool; "1. DSA truly sparse": chunking by query
 * does not change what is computed).  q_I: [L, Hi, di]; kpool: [P, di];
 * w: [L, Hi]; scores: [nrows, P], entries p >= elig(t) set to NaN. */
void oracle_indexer_scores(int64_t L, int32_t Hi, int32_t di,
                           const float *q_I, const float *kpool, const float *w,
                           const int64_t *rows, int64_t nrows, double *scores)
{
    int64_t P = L / 4;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows[r];
        int64_t e = elig(t);
        for (int64_t p = 0; p < P; ++p) {
            if (p >= e) {
                scores[r * P + p] = NAN;
                continue;
            }
            double s = 0.0;
            for (int32_t h = 0; h < Hi; ++h) {
                double dot = 0.0;
                for (int32_t i = 0; i < di; ++i)
                    dot += (double)q_I[(t * Hi + h) * di + i] * (double)kpool[p * di + i];
                double relu = dot > 0.0 ? dot : 0.0;
                s += (double)w[t * Hi + h] * relu;
            }
            scores[r * P + p] = s;
        }
    }
}

typedef struct { double s; int64_t p; } scored_pool;

/* Total order: higher score first; equal scores (including -0 == +0) go to
 * the lower pool index. */
static int by_score_then_index(const void *a, const void *b)
{
    const scored_pool *x = (const scored_pool *)a, *y = (const scored_pool *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    if (x->p < y->p) return -1;
    if (x->p > y->p) return 1;
    return 0;
}

static int by_int32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Per-query top-k pool selection (page 1, "Model and bottleneck": about 2048
 * keys read per query = 512 pools of 4).  scores: [nrows, P] as produced by
 * oracle_indexer_scores for the same rows; idx: [nrows, k]. */
int oracle_topk(int64_t L, int32_t k, const double *scores,
                const int64_t *rows, int64_t nrows, int32_t *idx)
{
    int64_t P = L / 4;
    scored_pool *buf = (scored_pool *)malloc((size_t)(P > 0 ? P : 1) * sizeof(scored_pool));
    if (!buf) return ORACLE_NO_MEMORY;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t e = elig(rows[r]);
        for (int64_t p = 0; p < e; ++p) {
            buf[p].s = scores[r * P + p];
            buf[p].p = p;
        }
        qsort(buf, (size_t)e, sizeof(scored_pool), by_score_then_index);
        int64_t m = e < k ? e : k;
        int32_t *out = idx + r * k;
        for (int64_t i = 0; i < m; ++i) out[i] = (int32_t)buf[i].p;
        qsort(out, (size_t)m, sizeof(int32_t), by_int32);
        for (int64_t i = m; i < k; ++i) out[i] = -1;
    }
    free(buf);
    return ORACLE_OK;
}

/* Tokens attended by query t: the selected pools' tokens (in the order idx
 * lists them), then the query's own partial pool when t mod 4 != 3 (page 1,
 * "1. DSA truly sparse": 2051 = 4*512 + 3 keys at most).  Returns the key
 * count, or -1 when idx names a pool the query may not see. */
int64_t oracle_key_set(int64_t t, const int32_t *idx_row, int32_t k, int64_t *keys)
{
    int64_t n = 0, e = elig(t);
    for (int32_t i = 0; i < k; ++i) {
        int64_t p = idx_row[i];
        if (p < 0) continue;
        if (p >= e) return -1;
        for (int j = 0; j < 4; ++j) keys[n++] = 4 * p + j;
    }
    if (t % 4 != 3)
        for (int64_t j = 4 * (t / 4); j <= t; ++j) keys[n++] = j;
    return n;
}

/* Sparse attention forward for the listed rows.  Q: [L, Hq, d], or
 * [nrows, Hq, d] holding only the listed rows when q_compact != 0;
 * K, V: [L, d]; idx: [L, k]; O: [nrows, Hq, d]; LSE: [nrows, Hq]. */
int oracle_attn_fwd(int64_t L, int32_t Hq, int32_t d, double scale,
                    const float *Q, int32_t q_compact, const float *K, const float *V,
                    const int32_t *idx, int32_t k,
                    const int64_t *rows, int64_t nrows, double *O, double *LSE)
{
    (void)L;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(4 * k + 4));
    double *s = (double *)malloc(sizeof(double) * (size_t)(4 * k + 4));
    if (!keys || !s) { free(keys); free(s); return ORACLE_NO_MEMORY; }
    int rc = ORACLE_OK;
    for (int64_t r = 0; r < nrows && rc == ORACLE_OK; ++r) {
        int64_t t = rows[r];
        int64_t n = oracle_key_set(t, idx + t * k, k, keys);
        if (n < 0) { rc = ORACLE_BAD_INDEX; break; }
        for (int32_t h = 0; h < Hq; ++h) {
            const float *q = Q + ((q_compact ? r : t) * Hq + h) * d;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int32_t i = 0; i < d; ++i) dot += (double)q[i] * (double)K[keys[j] * d + i];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
            double *o = O + (r * Hq + h) * d;
            for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double pj = exp(s[j] - m) / l;
                for (int32_t i = 0; i < d; ++i) o[i] += pj * (double)V[keys[j] * d + i];
            }
            LSE[r * Hq + h] = m + log(l);
        }
    }
    free(keys);
    free(s);
    return rc;
}

/* Sparse attention backward for the listed rows, given the upstream gradient
 * dO: [L, Hq, d] (Q and dO hold only the listed rows, [nrows, Hq, d], when
 * q_compact != 0).  Writes dQ: [nrows, Hq, d]; when dK and dV ([L, d]) are not
 * NULL, ADDS this rows' contributions to them (the caller zeroes them, and
 * may sum several disjoint row sets).  Uses its own double-precision O and
 * LSE.  No gradient flows to the indexer inputs. */
int oracle_attn_bwd(int64_t L, int32_t Hq, int32_t d, double scale,
                    const float *Q, int32_t q_compact, const float *K, const float *V,
                    const int32_t *idx, int32_t k, const float *dO,
                    const int64_t *rows, int64_t nrows,
                    double *dQ, double *dK, double *dV)
{
    (void)L;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(4 * k + 4));
    double *P = (double *)malloc(sizeof(double) * (size_t)(4 * k + 4));
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    if (!keys || !P || !o) { free(keys); free(P); free(o); return ORACLE_NO_MEMORY; }
    int rc = ORACLE_OK;
    for (int64_t r = 0; r < nrows && rc == ORACLE_OK; ++r) {
        int64_t t = rows[r];
        int64_t n = oracle_key_set(t, idx + t * k, k, keys);
        if (n < 0) { rc = ORACLE_BAD_INDEX; break; }
        for (int32_t h = 0; h < Hq; ++h) {
            const int64_t qr = q_compact ? r : t;
            const float *q = Q + (qr * Hq + h) * d;
            const float *go = dO + (qr * Hq + h) * d;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int32_t i = 0; i < d; ++i) dot += (double)q[i] * (double)K[keys[j] * d + i];
                P[j] = scale * dot;
                if (P[j] > m) m = P[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) l += exp(P[j] - m);
            for (int64_t j = 0; j < n; ++j) P[j] = exp(P[j] - m) / l;
            for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
            for (int64_t j = 0; j < n; ++j)
                for (int32_t i = 0; i < d; ++i) o[i] += P[j] * (double)V[keys[j] * d + i];
            double D = 0.0;
            for (int32_t i = 0; i < d; ++i) D += (double)go[i] * o[i];
            double *gq = dQ + (r * Hq + h) * d;
            for (int32_t i = 0; i < d; ++i) gq[i] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const float *kj = K + keys[j] * d, *vj = V + keys[j] * d;
                double dP = 0.0;
                for (int32_t i = 0; i < d; ++i) dP += (double)go[i] * (double)vj[i];
                double dS = P[j] * (dP - D);
                for (int32_t i = 0; i < d; ++i) gq[i] += scale * dS * (double)kj[i];
                if (dK && dV) {
                    for (int32_t i = 0; i < d; ++i) {
                        dK[keys[j] * d + i] += scale * dS * (double)q[i];
                        dV[keys[j] * d + i] += P[j] * (double)go[i];
                    }
                }
            }
        }
    }
    free(keys);
    free(P);
    free(o);
    return rc;
}
