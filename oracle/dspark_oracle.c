/*
 * dspark_oracle.c -- plain, slow CPU oracle for draft sampling and target
 * verification with the dyadic24-standard-v1 categorical q.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; every constant below is typed here from its definition.
 *
 * Sources (page title, section):
 *   [TR-dist]  "PP1 q transport and scheduling design", section
 *              "Distribution contract and precision" (dyadic q with M = 2^24,
 *              proposal construction, sparse top-k, integer draw, target p,
 *              ratio tests and full-vocabulary residual).
 *   [TR-v2]    same page, "Versioned v2 message design" (validation list,
 *              RNG ownership and separate acceptance / correction domains,
 *              commit = accepted count + correction/bonus IDs).
 *   [TR-shard] same page, "Sparse support and vocabulary-sharded TP2
 *              follow-up" (residual max(p - q, 0) over every token).
 *   [CONTRACT] "Remote DSpark drafter -- wire and state contract", section 2
 *              (anchor-as-first block; greedy argmax, lowest index on ties).
 *   [ATOM]     "DeepSeek-V4.1 DSpark", "State and sampling contracts"
 *              (greedy verification matches the target argmax; the verifier
 *              stops at the first mismatch).
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *              easy as 1, 2, 3", SC'11.
 *   Range reduction of exp: Cody and Waite, "Software Manual for the
 *              Elementary Functions" (1980): n = rint(d / ln2), r = d - n*ln2
 *              with ln2 split in a short high part and a low correction.
 *
 * Readings of points the pages leave open are stated at each function (the
 * same list is kept with the build's design notes).  All floating point here
 * is IEEE-754 round-to-nearest-even; the file must be compiled without
 * -ffast-math and with -ffp-contract=off so that every fp32 operation is the
 * single rounded operation written.
 *
 * Parity status: every exported function is pinned by tests that do not
 * re-type its formula (closed forms, exhaustive enumeration, library
 * cross-checks, an independent rational re-derivation on tiny vocabularies).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- status codes (oracle's own copy) ---------------------------------- */
enum {
    OR_OK = 0,
    OR_NONFINITE = 1,          /* NaN or +inf logit                          */
    OR_ZERO_MASS = 2,          /* no finite logit / empty support            */
    OR_ALLOC_INCONSISTENT = 3, /* remaining tickets out of range, sum != M   */
    OR_BAD_TEMPERATURE = 4,    /* T not finite, T <= 0, 1/T not normal       */
    OR_BAD_Q = 5,              /* sum of counts != M, non-canonical sparse   */
    OR_BAD_DRAFT = 6           /* draft id out of range or q(x) == 0         */
};

/* verification flags (per request) */
enum {
    OR_FLAG_AMBIG_ACCEPT = 1u,   /* |u*q - p| <= 1e-6 * q at a tested row    */
    OR_FLAG_NEAR_BOUNDARY = 2u,  /* draw within 1e-6 of a cumulative edge     */
    OR_FLAG_DEGENERATE = 4u,     /* residual mass <= 0, drew from p instead   */
    OR_FLAG_NEAR_BOUNDARY_REL = 8u /* draw within 1e-6 of an edge of its own
                                    token's interval, in units of that
                                    interval's width                         */
};

#define OR_M 16777216u                 /* 2^24 */
#define OR_PURPOSE_PROPOSAL 0u
#define OR_PURPOSE_ACCEPT 1u
#define OR_PURPOSE_RESIDUAL 2u
#define OR_PURPOSE_BONUS 3u

/* =========================================================================
 * Philox4x32-10 (SC'11).  Round: two 32x32->64 products of counter words 0
 * and 2 with the multipliers 0xD2511F53 and 0xCD9E8D57; the new counter is
 * (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0).  The key is bumped by the Weyl
 * constants 0x9E3779B9 / 0xBB67AE85 between rounds.  Ten rounds.
 * ========================================================================= */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4])
{
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k[2] = {key_in[0], key_in[1]};
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c[1] ^ k[0];
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c[3] ^ k[1];
        uint32_t n3 = lo0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    }
    out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

/* RNG key and counter layout of this library (reading of [TR-v2]: "keyed by
 * request generation, round, absolute predicted position, domain and draw
 * counter"): key = (seed low 32, seed high 32); counter = (request id, row,
 * purpose, 0).  The caller folds generation and round into the seed or the
 * request id.  One draw uses word 0 of the output. */
uint32_t oracle_draw_u32(uint64_t seed, uint32_t request, uint32_t row,
                         uint32_t purpose)
{
    uint32_t ctr[4] = {request, row, purpose, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[0];
}

/* =========================================================================
 * exp_ds: the deterministic fp32 exponential used to weight draft tokens.
 * [TR-dist] asks for globally normalised draft weights and exact, reproducible
 * integer counts but fixes no exp; this build fixes one (reading Q1):
 *   d >= -87 (else 0);  t = RN(d * L2E);  n = rint(t) (ties to even);
 *   r = fma(-n, LN2_HI, d);  r = fma(-n, LN2_LO, r);
 *   p = Horner form of the degree-7 Taylor polynomial of e^r, one fma a step;
 *   result = p * 2^n (exact: the result is a normal float on this domain).
 * Constants: L2E = float nearest 1/ln2; LN2_HI = ln2 truncated to 16 bits
 * after the binary point (so n * LN2_HI is exact for |n| <= 127);
 * LN2_LO = float nearest (ln2 - LN2_HI); C_k = float nearest 1/k!.
 * ========================================================================= */
static const float OR_L2E = 0x1.715476p+0f;
static const float OR_LN2_HI = 0x1.62e4p-1f;
static const float OR_LN2_LO = 0x1.7f7d1cp-20f;
static const float OR_C2 = 0x1p-1f;
static const float OR_C3 = 0x1.555556p-3f;
static const float OR_C4 = 0x1.555556p-5f;
static const float OR_C5 = 0x1.111112p-7f;
static const float OR_C6 = 0x1.6c16c2p-10f;
static const float OR_C7 = 0x1.a01a02p-13f;

float oracle_exp_ds(float d)
{
    if (!(d >= -87.0f)) return 0.0f;
    float t = d * OR_L2E;
    float n = rintf(t);
    float r = fmaf(-n, OR_LN2_HI, d);
    r = fmaf(-n, OR_LN2_LO, r);
    float p = OR_C7;
    p = fmaf(p, r, OR_C6);
    p = fmaf(p, r, OR_C5);
    p = fmaf(p, r, OR_C4);
    p = fmaf(p, r, OR_C3);
    p = fmaf(p, r, OR_C2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return ldexpf(p, (int)n);
}

void oracle_exp_ds_array(const float* d, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_exp_ds(d[i]);
}

/* =========================================================================
 * q construction, step 1-4 ([TR-dist] "Proposal construction"): validate,
 * apply temperature, choose the support, integer weights E_v and their sum.
 *   invT = RN32(1/T);  y_v = RN32(x_v * invT)                    (reading Q4)
 *   dense support: every y_v > -inf;  top-k support: the k largest y_v,
 *   ties to the lowest id, all finite entries if fewer than k    (reading Q6)
 *   m = max over the support;  d_v = RN32(y_v - m);  e_v = exp_ds(d_v)
 *   E_v = floor(e_v * 2^40) (exact);  S = sum of E_v in uint64  (reading Q2)
 * `E` gets E_v on the support and 0 elsewhere; `in_support` 1/0 per token.
 * ========================================================================= */
typedef struct { float y; int32_t id; } or_yid;

static int or_cmp_topk(const void* a, const void* b)
{
    const or_yid* u = (const or_yid*)a;
    const or_yid* v = (const or_yid*)b;
    if (u->y > v->y) return -1;
    if (u->y < v->y) return 1;
    return (u->id < v->id) ? -1 : (u->id > v->id) ? 1 : 0;
}

int oracle_q_weights_row(const float* x, int32_t V, float T, int32_t top_k,
                         uint64_t* E, uint8_t* in_support, uint64_t* S_out)
{
    memset(E, 0, sizeof(uint64_t) * (size_t)V);
    memset(in_support, 0, (size_t)V);
    if (S_out) *S_out = 0;
    if (!(isfinite(T) && T > 0.0f)) return OR_BAD_TEMPERATURE;
    float invT = 1.0f / T;
    if (!(isfinite(invT) && invT >= 0x1p-126f)) return OR_BAD_TEMPERATURE;

    float* y = (float*)malloc(sizeof(float) * (size_t)V);
    if (!y) return -1;
    int32_t n_finite = 0;
    for (int32_t v = 0; v < V; ++v) {
        float xv = x[v];
        if (isnan(xv) || xv == INFINITY) { free(y); return OR_NONFINITE; }
        float yv = xv * invT;
        if (isfinite(xv) && !isfinite(yv)) { free(y); return OR_NONFINITE; }
        y[v] = yv;
        if (yv > -INFINITY) ++n_finite;
    }
    if (n_finite == 0) { free(y); return OR_ZERO_MASS; }

    if (top_k > 0 && top_k < n_finite) {
        or_yid* list = (or_yid*)malloc(sizeof(or_yid) * (size_t)n_finite);
        if (!list) { free(y); return -1; }
        int32_t j = 0;
        for (int32_t v = 0; v < V; ++v)
            if (y[v] > -INFINITY) { list[j].y = y[v]; list[j].id = v; ++j; }
        qsort(list, (size_t)n_finite, sizeof(or_yid), or_cmp_topk);
        for (int32_t i = 0; i < top_k; ++i) in_support[list[i].id] = 1;
        free(list);
    } else {
        for (int32_t v = 0; v < V; ++v) in_support[v] = (y[v] > -INFINITY);
    }

    float m = -INFINITY;
    for (int32_t v = 0; v < V; ++v)
        if (in_support[v] && y[v] > m) m = y[v];

    uint64_t S = 0;
    for (int32_t v = 0; v < V; ++v) {
        if (!in_support[v]) continue;
        float d = y[v] - m;
        float e = oracle_exp_ds(d);
        uint64_t Ev = (uint64_t)floor((double)e * 1099511627776.0); /* 2^40 */
        E[v] = Ev;
        S += Ev;
    }
    free(y);
    if (S_out) *S_out = S;
    return OR_OK;
}

/* =========================================================================
 * q construction, steps 5-7: FP64 floor plus largest remainders.
 *   k = RN64(2^24 / RN64(S));  a_v = RN64(E_v * k)               (reading Q3)
 *   f_v = floor(a_v);  r_v = a_v - f_v (both exact in FP64)
 *   F = sum f_v;  R = M - F;  require 0 <= R < M and R <= #{r_v > 0}
 *   grant +1 to the R support tokens with the largest r_v, ties to the lowest
 *   id;  c_v = f_v + grant;  require sum c_v == M in uint64.
 * Refuse (ALLOC_INCONSISTENT, counts all zero) rather than clip.
 * ========================================================================= */
typedef struct { double r; int32_t id; } or_rid;

static int or_cmp_remainder(const void* a, const void* b)
{
    const or_rid* u = (const or_rid*)a;
    const or_rid* v = (const or_rid*)b;
    if (u->r > v->r) return -1;
    if (u->r < v->r) return 1;
    return (u->id < v->id) ? -1 : (u->id > v->id) ? 1 : 0;
}

int oracle_q_allocate_row(const uint64_t* E, const uint8_t* in_support,
                          int32_t V, uint32_t* counts)
{
    memset(counts, 0, sizeof(uint32_t) * (size_t)V);
    uint64_t S = 0;
    int32_t n_support = 0;
    for (int32_t v = 0; v < V; ++v)
        if (in_support[v]) { S += E[v]; ++n_support; }
    if (n_support == 0 || S == 0) return OR_ZERO_MASS;

    double k = 16777216.0 / (double)S;
    or_rid* rem = (or_rid*)malloc(sizeof(or_rid) * (size_t)n_support);
    if (!rem) return -1;
    uint64_t F = 0;
    int32_t n_rem = 0, n_positive = 0;
    for (int32_t v = 0; v < V; ++v) {
        if (!in_support[v]) continue;
        double a = (double)E[v] * k;
        double f = floor(a);
        double r = a - f;
        counts[v] = (uint32_t)f;
        F += (uint64_t)f;
        rem[n_rem].r = r;
        rem[n_rem].id = v;
        ++n_rem;
        if (r > 0.0) ++n_positive;
    }
    if (F > (uint64_t)OR_M) {
        memset(counts, 0, sizeof(uint32_t) * (size_t)V);
        free(rem);
        return OR_ALLOC_INCONSISTENT;
    }
    uint64_t R = (uint64_t)OR_M - F;
    if (R >= (uint64_t)OR_M || R > (uint64_t)n_positive) {
        memset(counts, 0, sizeof(uint32_t) * (size_t)V);
        free(rem);
        return OR_ALLOC_INCONSISTENT;
    }
    qsort(rem, (size_t)n_rem, sizeof(or_rid), or_cmp_remainder);
    for (uint64_t i = 0; i < R; ++i) counts[rem[i].id] += 1u;
    free(rem);

    uint64_t total = 0;
    for (int32_t v = 0; v < V; ++v) total += counts[v];
    if (total != (uint64_t)OR_M) {
        memset(counts, 0, sizeof(uint32_t) * (size_t)V);
        return OR_ALLOC_INCONSISTENT;
    }
    return OR_OK;
}

/* Whole q build for one row.  Dense (top_k == 0): counts[V].  Sparse
 * (top_k > 0): the nonzero counts in ascending id order in ids[]/counts[]
 * (capacity top_k), *nnz entries, the rest of the capacity id -1 / count 0
 * ([TR-dist]: "Drop zero-count entries and declare zero everywhere else").
 * On a refused row every count is 0 (and *nnz = 0). */
int oracle_q_build_row(const float* x, int32_t V, float T, int32_t top_k,
                       uint32_t* counts, int32_t* ids, int32_t* nnz)
{
    uint64_t* E = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
    uint8_t* sup = (uint8_t*)malloc((size_t)V);
    uint32_t* dense = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)V);
    if (!E || !sup || !dense) { free(E); free(sup); free(dense); return -1; }
    int st = oracle_q_weights_row(x, V, T, top_k, E, sup, NULL);
    if (st == OR_OK) st = oracle_q_allocate_row(E, sup, V, dense);
    if (st != OR_OK) memset(dense, 0, sizeof(uint32_t) * (size_t)V);
    if (top_k > 0) {
        int32_t j = 0;
        for (int32_t i = 0; i < top_k; ++i) { ids[i] = -1; counts[i] = 0; }
        for (int32_t v = 0; v < V && st == OR_OK; ++v) {
            if (dense[v] == 0) continue;
            if (j >= top_k) { st = OR_ALLOC_INCONSISTENT; break; }
            ids[j] = v; counts[j] = dense[v]; ++j;
        }
        if (st != OR_OK) {
            for (int32_t i = 0; i < top_k; ++i) { ids[i] = -1; counts[i] = 0; }
            j = 0;
        }
        *nnz = j;
    } else {
        memcpy(counts, dense, sizeof(uint32_t) * (size_t)V);
        if (nnz) *nnz = 0;
    }
    free(E); free(sup); free(dense);
    return st;
}

/* Batched q build: rows r = 0..n_rows-1 at x + r*ld; temperature[r] (or 1.0
 * if temperature == NULL).  Dense counts at counts + r*V; sparse at
 * ids/counts + r*top_k and nnz[r]. */
void oracle_q_build(const float* x, int64_t ld, int32_t n_rows, int32_t V,
                    const float* temperature, int32_t top_k, uint32_t* counts,
                    int32_t* ids, int32_t* nnz, int32_t* status)
{
    for (int32_t r = 0; r < n_rows; ++r) {
        float T = temperature ? temperature[r] : 1.0f;
        if (top_k > 0)
            status[r] = oracle_q_build_row(x + (int64_t)r * ld, V, T, top_k,
                                           counts + (int64_t)r * top_k,
                                           ids + (int64_t)r * top_k, nnz + r);
        else
            status[r] = oracle_q_build_row(x + (int64_t)r * ld, V, T, 0,
                                           counts + (int64_t)r * V, NULL, NULL);
    }
}

/* =========================================================================
 * Integer categorical draw ([TR-dist]: "a uniform 24-bit integer and exact
 * integer cumulative counts (first cumulative count strictly greater than
 * the draw)").  Walks the entries in ascending id order.
 * n entries; ids == NULL means entry i is token i.  Returns -1 if no entry
 * qualifies (only possible when the counts do not sum above D).
 * ========================================================================= */
int32_t oracle_categorical_pick(const uint32_t* counts, const int32_t* ids,
                                int32_t n, uint32_t D)
{
    uint64_t cum = 0;
    for (int32_t i = 0; i < n; ++i) {
        cum += counts[i];
        if (cum > (uint64_t)D) return ids ? ids[i] : i;
    }
    return -1;
}

void oracle_categorical_pick_many(const uint32_t* counts, const int32_t* ids,
                                  int32_t n, const uint32_t* D, int64_t n_draws,
                                  int32_t* out)
{
    for (int64_t t = 0; t < n_draws; ++t)
        out[t] = oracle_categorical_pick(counts, ids, n, D[t]);
}

/* Draft sample: D = (philox(seed; request, row, PROPOSAL) word 0) >> 8, the
 * top 24 bits of the 32-bit draw (reading Q7).  A row whose counts do not
 * sum to M, or a sparse row (ids != NULL) that is not canonical -- at least
 * one entry, ids strictly ascending in [0, V), every count > 0 -- is refused
 * (BAD_Q, token -1), following the validation list of [TR-v2]. */
int32_t oracle_draft_sample_row(const uint32_t* counts, const int32_t* ids,
                                int32_t n, int32_t V, uint64_t seed,
                                uint32_t request, uint32_t row, int32_t* status)
{
    uint64_t total = 0;
    if (ids) {
        if (n < 1) { *status = OR_BAD_Q; return -1; }
        for (int32_t i = 0; i < n; ++i) {
            if (ids[i] < 0 || ids[i] >= V || counts[i] == 0 ||
                (i > 0 && ids[i] <= ids[i - 1])) {
                *status = OR_BAD_Q;
                return -1;
            }
        }
    }
    for (int32_t i = 0; i < n; ++i) total += counts[i];
    if (total != (uint64_t)OR_M) { *status = OR_BAD_Q; return -1; }
    uint32_t D = oracle_draw_u32(seed, request, row, OR_PURPOSE_PROPOSAL) >> 8;
    *status = OR_OK;
    return oracle_categorical_pick(counts, ids, n, D);
}

/* =========================================================================
 * Target p ([TR-dist]: "the distribution after the unchanged target
 * processors, penalties, grammar, T=1 and top_p=1"), FP64 with libm exp:
 *   m = max z;  p_v = exp(z_v - m) / sum_u exp(z_u - m);  -inf -> 0.
 * NaN / +inf -> NONFINITE; no finite logit -> ZERO_MASS.
 * Also the greedy argmax: the lowest id among the maxima ([CONTRACT] s.2).
 * ========================================================================= */
int oracle_target_row(const float* z, int32_t V, double* p, int32_t* argmax)
{
    int32_t am = -1;
    float m = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        float zv = z[v];
        if (isnan(zv) || zv == INFINITY) return OR_NONFINITE;
        if (zv > m) { m = zv; am = v; }
    }
    if (am < 0) return OR_ZERO_MASS;
    if (argmax) *argmax = am;
    if (p) {
        double s = 0.0;
        for (int32_t v = 0; v < V; ++v) {
            double e = (z[v] == -INFINITY) ? 0.0 : exp((double)z[v] - (double)m);
            p[v] = e;
            s += e;
        }
        for (int32_t v = 0; v < V; ++v) p[v] /= s;
    }
    return OR_OK;
}

void oracle_target_probs(const float* z, int64_t ld, int32_t n_rows, int32_t V,
                         double* p, int32_t* argmax, int32_t* status)
{
    for (int32_t r = 0; r < n_rows; ++r) {
        int32_t am = -1;
        status[r] = oracle_target_row(z + (int64_t)r * ld, V,
                                      p ? p + (int64_t)r * V : NULL, &am);
        if (argmax) argmax[r] = (status[r] == OR_OK) ? am : -1;
    }
}

/* =========================================================================
 * Ratio test (reading Q9 of [TR-dist] "Ratio tests"): accept draft x_j with
 * probability min(1, p/q):  u = U * 2^-24 with U the 24-bit acceptance draw,
 * q = c / 2^24;  accept  <=>  u * q < p  <=>  U * c < p * 2^48 (strict).
 * U * c is an exact integer < 2^48; p * 2^48 is an exact scaling.
 * ========================================================================= */
int oracle_ratio_accept(uint32_t U, uint32_t c, double p)
{
    double lhs = (double)((uint64_t)U * (uint64_t)c);
    return lhs < p * 281474976710656.0; /* 2^48 */
}

void oracle_ratio_accept_many(const uint32_t* U, int64_t n, uint32_t c,
                              double p, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_ratio_accept(U[i], c, p);
}

/* =========================================================================
 * Residual / bonus pick ([TR-dist] "full-vocabulary residual sampling";
 * [TR-shard] "max(p-q,0) for every token").  With c == NULL the weights are p
 * itself (bonus draw).  w is a 32-bit draw; t = (w * 2^-32) * Z; the token is
 * the first v (ascending id) whose cumulative weight exceeds t (reading Q13):
 *   Z <= 0 -> draw from p instead (flag DEGENERATE);
 *   t beyond the rounded total -> the last token with positive weight;
 *   NEAR_BOUNDARY if t lies within 1e-6 (probability units) of either edge
 *   of the chosen token's cumulative interval;
 *   NEAR_BOUNDARY_REL if it lies within 1e-6 * r_pick of either edge, r_pick
 *   the chosen token's own weight: the draw's position inside its token's
 *   interval is within 1e-6 of an end, as the ratio test's band
 *   |u*q - p| <= 1e-6*q is relative to q.  This band is contained in the
 *   absolute one (r_pick <= 1) and a uniform t falls in it with probability
 *   2e-6 whatever the row.
 * ========================================================================= */
int32_t oracle_residual_pick(const double* p, const uint32_t* c, int32_t V,
                             uint32_t w, uint32_t* flags)
{
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r) return -1;
    double Z = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double q = c ? (double)c[v] / 16777216.0 : 0.0;
        double rv = p[v] - q;
        r[v] = rv > 0.0 ? rv : 0.0;
        Z += r[v];
    }
    if (!(Z > 0.0)) {
        if (flags) *flags |= OR_FLAG_DEGENERATE;
        Z = 0.0;
        for (int32_t v = 0; v < V; ++v) { r[v] = p[v]; Z += r[v]; }
    }
    double t = ((double)w * 0x1p-32) * Z;
    double cum = 0.0, prev = 0.0;
    int32_t pick = -1, last_pos = -1;
    for (int32_t v = 0; v < V; ++v) {
        if (r[v] > 0.0) last_pos = v;
        prev = cum;
        cum += r[v];
        if (cum > t) { pick = v; break; }
    }
    if (pick < 0) {
        pick = last_pos;
        prev = cum - (last_pos >= 0 ? r[last_pos] : 0.0);
    }
    if (flags && (fabs(t - prev) <= 1e-6 || fabs(cum - t) <= 1e-6))
        *flags |= OR_FLAG_NEAR_BOUNDARY;
    if (flags && pick >= 0 &&
        (fabs(t - prev) <= 1e-6 * r[pick] || fabs(cum - t) <= 1e-6 * r[pick]))
        *flags |= OR_FLAG_NEAR_BOUNDARY_REL;
    free(r);
    return pick;
}

/* ---- helpers for the verifiers ----------------------------------------- */

/* q row j as dense counts.  Dense: a pointer into counts.  Sparse: expands
 * the (id, count) list into `scratch` after checking its canonical form
 * ([TR-v2]: reject duplicate, unsorted, out-of-range ids, zero or missing
 * entries, wrong total mass).  Returns OR_OK or OR_BAD_Q. */
static int or_q_row(const uint32_t* counts, const int32_t* ids,
                    const int32_t* nnz, int32_t top_k, int32_t V, int64_t row,
                    uint32_t* scratch, const uint32_t** out)
{
    if (top_k == 0) {
        *out = counts + row * (int64_t)V;
        return OR_OK;
    }
    const int32_t* id = ids + row * (int64_t)top_k;
    const uint32_t* cn = counts + row * (int64_t)top_k;
    int32_t n = nnz[row];
    memset(scratch, 0, sizeof(uint32_t) * (size_t)V);
    *out = scratch;
    if (n < 1 || n > top_k) return OR_BAD_Q;
    uint64_t total = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (id[i] < 0 || id[i] >= V) return OR_BAD_Q;
        if (i > 0 && id[i] <= id[i - 1]) return OR_BAD_Q;
        if (cn[i] == 0) return OR_BAD_Q;
        scratch[id[i]] = cn[i];
        total += cn[i];
    }
    if (total != (uint64_t)OR_M) return OR_BAD_Q;
    return OR_OK;
}

static void or_discard(int32_t depth, int32_t* accept_len, int32_t* committed)
{
    *accept_len = 0;
    for (int32_t i = 0; i <= depth; ++i) committed[i] = -1;
}

/* =========================================================================
 * Greedy verification of one request ([ATOM]: "Greedy verification matches
 * target argmax"; [CONTRACT] s.2 anchor-as-first block: target row j scores
 * the token drafted at position j, row `depth` gives the bonus).  Rows are
 * read in order and the verifier stops at the first mismatch, so a row after
 * it is never read or validated.
 *   L = first j with x_j != argmax_j, else depth;
 *   committed = x_0 .. x_{L-1}, argmax_L;  the rest -1.
 * Bad request (status != OK): accept_len 0, committed all -1.
 * ========================================================================= */
int oracle_verify_greedy_req(const float* z, int64_t ld, int32_t V,
                             int32_t depth, const int32_t* drafts,
                             int32_t* accept_len, int32_t* committed)
{
    or_discard(depth, accept_len, committed);
    for (int32_t j = 0; j < depth; ++j)
        if (drafts[j] < 0 || drafts[j] >= V) return OR_BAD_DRAFT;
    int32_t L = depth, last = -1;
    for (int32_t j = 0; j <= depth; ++j) {
        int32_t am = -1;
        int st = oracle_target_row(z + (int64_t)j * ld, V, NULL, &am);
        if (st != OR_OK) { or_discard(depth, accept_len, committed); return st; }
        if (j == depth || am != drafts[j]) { L = j; last = am; break; }
    }
    *accept_len = L;
    for (int32_t i = 0; i < L; ++i) committed[i] = drafts[i];
    committed[L] = last;
    return OR_OK;
}

/* =========================================================================
 * Standard ratio verification of one request ([TR-dist], [TR-v2], [TR-shard]
 * and reading Q9-Q13).  For j = 0, 1, ... (stopping at the first rejection):
 *   target row j -> p_j (FP64);  q row j -> c_j (sparse rows checked
 *   canonical);  c_j(x_j) == 0 -> BAD_DRAFT;
 *   U_j = (philox(seed; request, j, ACCEPT) word 0) >> 8;
 *   accept <=> U_j * c_j(x_j) < p_j(x_j) * 2^48.
 * First rejection at L < depth: dense q row L must sum to M (BAD_Q), then the
 * correction token is drawn from max(p_L - q_L, 0) over all V with
 * w = philox(seed; request, L, RESIDUAL) word 0.
 * All accepted: the bonus token is drawn from p_depth with
 * w = philox(seed; request, depth, BONUS) word 0.
 * committed = x_0 .. x_{L-1}, correction-or-bonus; the rest -1.
 * flags: AMBIG_ACCEPT if |U*c*2^-48 - p| <= 1e-6 * c * 2^-24 at a tested
 * row; NEAR_BOUNDARY / DEGENERATE from the final pick.
 * ========================================================================= */
int oracle_verify_ratio_req(const float* z, int64_t ld, int32_t V,
                            int32_t depth, const int32_t* drafts,
                            const uint32_t* counts, const int32_t* ids,
                            const int32_t* nnz, int32_t top_k, uint64_t seed,
                            uint32_t request, int32_t* accept_len,
                            int32_t* committed, uint32_t* flags)
{
    uint32_t fl = 0;
    or_discard(depth, accept_len, committed);
    if (flags) *flags = 0;
    for (int32_t j = 0; j < depth; ++j)
        if (drafts[j] < 0 || drafts[j] >= V) return OR_BAD_DRAFT;

    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    uint32_t* scratch = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)V);
    if (!p || !scratch) { free(p); free(scratch); return -1; }

    int st = OR_OK;
    int32_t L = depth, pick = -1;
    for (int32_t j = 0; j < depth; ++j) {
        st = oracle_target_row(z + (int64_t)j * ld, V, p, NULL);
        if (st != OR_OK) goto done;
        const uint32_t* q = NULL;
        st = or_q_row(counts, ids, nnz, top_k, V, (int64_t)j, scratch, &q);
        if (st != OR_OK) goto done;
        uint32_t c = q[drafts[j]];
        if (c == 0) { st = OR_BAD_DRAFT; goto done; }
        uint32_t U = oracle_draw_u32(seed, request, (uint32_t)j, OR_PURPOSE_ACCEPT) >> 8;
        double pj = p[drafts[j]];
        double uq = (double)((uint64_t)U * (uint64_t)c) * 0x1p-48;
        if (fabs(uq - pj) <= 1e-6 * ((double)c * 0x1p-24)) fl |= OR_FLAG_AMBIG_ACCEPT;
        if (!oracle_ratio_accept(U, c, pj)) {
            L = j;
            if (top_k == 0) {
                uint64_t total = 0;
                for (int32_t v = 0; v < V; ++v) total += q[v];
                if (total != (uint64_t)OR_M) { st = OR_BAD_Q; goto done; }
            }
            uint32_t w = oracle_draw_u32(seed, request, (uint32_t)j, OR_PURPOSE_RESIDUAL);
            pick = oracle_residual_pick(p, q, V, w, &fl);
            break;
        }
    }
    if (L == depth) {
        st = oracle_target_row(z + (int64_t)depth * ld, V, p, NULL);
        if (st != OR_OK) goto done;
        uint32_t w = oracle_draw_u32(seed, request, (uint32_t)depth, OR_PURPOSE_BONUS);
        pick = oracle_residual_pick(p, NULL, V, w, &fl);
    }
    *accept_len = L;
    for (int32_t i = 0; i < L; ++i) committed[i] = drafts[i];
    committed[L] = pick;
done:
    if (st != OR_OK) { or_discard(depth, accept_len, committed); fl = 0; }
    if (flags) *flags = fl;
    free(p);
    free(scratch);
    return st;
}

/* =========================================================================
 * Received q: wire form, byte checksum and validation ("PP1 q transport and
 * scheduling design", Distribution contract and precision: q sent as
 * little-endian FP32 q = c / M, counts recovered by multiplying by M and
 * required to be integers, the mass checked in uint64; Versioned v2 message
 * design: per-position reply with q values, sparse ids and a checksum, and
 * the list of refusals).
 *
 * Readings (the pages fix no checksum algorithm and no sparse byte order):
 *   - payload words: dense row = the V FP32 bit patterns in id order;
 *     sparse row = the nnz int32 ids, then their nnz FP32 bit patterns;
 *   - byte checksum = Fletcher-64 of the payload words (A and B summed modulo
 *     2^32 - 1 from zero, checksum = B << 32 | A);
 *   - validation order: a sparse entry count outside [1, top_k] (BAD_Q: the
 *     payload's size), then the checksum (if one is given), then the row's
 *     values and support (BAD_Q), then the proposed token (BAD_DRAFT; a
 *     negative token is one outside [0, V)).
 * ========================================================================= */
#define OR_BAD_CHECKSUM 9

uint64_t oracle_fletcher64(const uint32_t* words, int64_t n)
{
    const uint64_t mod = 0xFFFFFFFFull;
    uint64_t a = 0, b = 0;
    for (int64_t i = 0; i < n; ++i) {
        a = (a + words[i]) % mod;
        b = (b + a) % mod;
    }
    return (b << 32) | a;
}

static uint32_t or_f32_bits(float v) { uint32_t u; memcpy(&u, &v, 4); return u; }

/* Wire form of one q row.  Dense (top_k == 0): q[v] = counts[v] / M for the
 * V ids.  Sparse: q[i] = counts[i] / M for the nnz entries, and q = 0 past
 * them.  Returns the checksum of the row's payload. */
uint64_t oracle_q_pack_row(const uint32_t* counts, const int32_t* ids, int32_t nnz,
                           int32_t top_k, int32_t V, float* q)
{
    int64_t n = top_k > 0 ? nnz : V;
    if (n < 0) n = 0;
    for (int64_t i = 0; i < n; ++i) q[i] = (float)((double)counts[i] / (double)OR_M);
    if (top_k > 0)
        for (int64_t i = n; i < top_k; ++i) q[i] = 0.0f;
    uint32_t* words = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(2 * n + 1));
    if (!words) return 0;
    int64_t w = 0;
    if (top_k > 0)
        for (int64_t i = 0; i < n; ++i) words[w++] = (uint32_t)ids[i];
    for (int64_t i = 0; i < n; ++i) words[w++] = or_f32_bits(q[i]);
    uint64_t cs = oracle_fletcher64(words, w);
    free(words);
    return cs;
}

/* Validation of one received q row.  counts_out (may be NULL) gets the
 * recovered counts (dense [V] or sparse [top_k], zeros past nnz and on a
 * refusal).  token: the proposed token, checked when has_token.  expect: the
 * checksum the row must have, checked when has_expect. */
int oracle_q_validate_row(const float* q, const int32_t* ids, int32_t nnz, int32_t top_k,
                          int32_t V, int has_token, int32_t token, int has_expect,
                          uint64_t expect, uint32_t* counts_out)
{
    int64_t cap = top_k > 0 ? top_k : V;
    if (counts_out) memset(counts_out, 0, sizeof(uint32_t) * (size_t)cap);
    if (top_k > 0 && (nnz < 1 || nnz > top_k)) return OR_BAD_Q;
    int64_t n = top_k > 0 ? nnz : V;
    if (has_expect) {
        uint32_t* words = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(2 * n + 1));
        if (!words) return -1;
        int64_t w = 0;
        if (top_k > 0)
            for (int64_t i = 0; i < n; ++i) words[w++] = (uint32_t)ids[i];
        for (int64_t i = 0; i < n; ++i) words[w++] = or_f32_bits(q[i]);
        uint64_t cs = oracle_fletcher64(words, w);
        free(words);
        if (cs != expect) return OR_BAD_CHECKSUM;
    }
    /* values: finite, not negative, dyadic (q * M an integer, at most M) */
    uint32_t* c = (uint32_t*)calloc((size_t)cap, sizeof(uint32_t));
    if (!c) return -1;
    uint64_t total = 0;
    int st = OR_OK;
    for (int64_t i = 0; i < n && st == OR_OK; ++i) {
        double v = (double)q[i];
        if (!isfinite(v) || v < 0.0) { st = OR_BAD_Q; break; }
        double cm = v * (double)OR_M;
        if (cm != floor(cm) || cm > (double)OR_M) { st = OR_BAD_Q; break; }
        c[i] = (uint32_t)cm;
        total += c[i];
        if (top_k > 0) {
            /* canonical support: ids strictly ascending in [0, V), no zero
             * entries listed */
            if (ids[i] < 0 || ids[i] >= V || c[i] == 0) st = OR_BAD_Q;
            if (i > 0 && ids[i - 1] >= ids[i]) st = OR_BAD_Q;
        }
    }
    if (st == OR_OK && total != (uint64_t)OR_M) st = OR_BAD_Q;
    if (st == OR_OK && has_token) {
        if (token < 0 || token >= V) st = OR_BAD_DRAFT;
        else if (top_k == 0) { if (c[token] == 0) st = OR_BAD_DRAFT; }
        else {
            int found = 0;
            for (int64_t i = 0; i < n; ++i) if (ids[i] == token) found = 1;
            if (!found) st = OR_BAD_DRAFT;
        }
    }
    if (st == OR_OK && counts_out) memcpy(counts_out, c, sizeof(uint32_t) * (size_t)cap);
    free(c);
    return st;
}

/* =========================================================================
 * Stochastic (match) verification ("DeepSeek-V4.1 DSpark", State and
 * sampling contracts): every verify row draws a token from the target's own
 * p with independent noise, a proposal is accepted when the draw equals it,
 * and verification stops at the first mismatch, committing that row's draw
 * (the draw of row depth when every proposal matched).  This keeps p's
 * distribution; it is not the ratio test.  Reading: the draw of row j uses
 * the purpose MATCH = 4 and the same inverse-CDF pick over p as the bonus
 * draw; refusals as in the other verifiers (draft ids up front, then each
 * row read).
 * ========================================================================= */
#define OR_PURPOSE_MATCH 4u

int oracle_verify_match_req(const float* z, int64_t ld, int32_t V, int32_t depth,
                            const int32_t* drafts, uint64_t seed, uint32_t request,
                            int32_t* accept_len, int32_t* committed, uint32_t* flags)
{
    uint32_t fl = 0;
    or_discard(depth, accept_len, committed);
    if (flags) *flags = 0;
    for (int32_t j = 0; j < depth; ++j)
        if (drafts[j] < 0 || drafts[j] >= V) return OR_BAD_DRAFT;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p) return -1;
    int st = OR_OK;
    int32_t L = depth, pick = -1;
    for (int32_t j = 0; j <= depth; ++j) {
        st = oracle_target_row(z + (int64_t)j * ld, V, p, NULL);
        if (st != OR_OK) break;
        uint32_t w = oracle_draw_u32(seed, request, (uint32_t)j, OR_PURPOSE_MATCH);
        int32_t t = oracle_residual_pick(p, NULL, V, w, &fl);
        if (j < depth && t == drafts[j]) continue;
        L = j;
        pick = t;
        break;
    }
    if (st == OR_OK) {
        *accept_len = L;
        for (int32_t i = 0; i < L; ++i) committed[i] = drafts[i];
        committed[L] = pick;
    } else {
        or_discard(depth, accept_len, committed);
        fl = 0;
    }
    if (flags) *flags = fl;
    free(p);
    return st;
}

/* =========================================================================
 * Markov-conditioned draft chain ("Remote DSpark drafter -- wire and state
 * contract", section 2: the sequential Markov step adds the bias row of the
 * previous sampled token to the base logits, the anchor at step 0; section
 * 6.3: the optional margin is top1 - top2 of (base + Markov) logits at each
 * step).  Readings: z_v = RN32(x_v + bias[prev mod n_bias][v]); the dense q
 * of z with the row's temperature, then the draft draw of that row; the
 * margin is z's largest finite value minus its second largest (equal values
 * give 0), FLT_MAX when fewer than two are finite, 0 for a refused row; a row
 * after a refused row is refused with the same status (the chain has no
 * token to condition on); an anchor outside [0, V) refuses the request with
 * BAD_DRAFT.
 * ========================================================================= */
int oracle_q_chain_request(const float* x, int64_t ld, int32_t V, int32_t depth,
                           const float* temperature, const float* bias, int64_t bias_ld,
                           int32_t n_bias, int32_t anchor, uint64_t seed, uint32_t request,
                           uint32_t* counts, int32_t* tokens, int32_t* status, float* margins)
{
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    if (!z) return -1;
    int32_t prev = anchor;
    int refused = (anchor < 0 || anchor >= V) ? OR_BAD_DRAFT : OR_OK;
    for (int32_t j = 0; j < depth; ++j) {
        uint32_t* c = counts + (int64_t)j * V;
        if (refused != OR_OK) {
            memset(c, 0, sizeof(uint32_t) * (size_t)V);
            tokens[j] = -1;
            status[j] = refused;
            if (margins) margins[j] = 0.0f;
            continue;
        }
        const float* xr = x + (int64_t)j * ld;
        const float* br = bias ? bias + (int64_t)(prev % n_bias) * bias_ld : NULL;
        float t1 = -INFINITY, t2 = -INFINITY;
        int32_t nfin = 0;
        for (int32_t v = 0; v < V; ++v) {
            z[v] = br ? xr[v] + br[v] : xr[v];
            if (isfinite(z[v])) {
                ++nfin;
                if (z[v] > t1) { t2 = t1; t1 = z[v]; }
                else if (z[v] > t2) t2 = z[v];
            }
        }
        float T = temperature ? temperature[j] : 1.0f;
        int32_t ids_unused = 0, nnz_unused = 0;
        int st = oracle_q_build_row(z, V, T, 0, c, &ids_unused, &nnz_unused);
        if (st == OR_OK) {
            int32_t st2 = OR_OK;
            tokens[j] = oracle_draft_sample_row(c, NULL, V, V, seed, request, (uint32_t)j, &st2);
            st = st2;
        }
        if (st != OR_OK) {
            tokens[j] = -1;
            refused = st;
        }
        status[j] = st;
        if (margins) {
            float mg = 0.0f;
            if (st == OR_OK) {
                if (nfin < 2) mg = FLT_MAX;
                else {
                    mg = t1 - t2;
                    if (!(mg <= FLT_MAX)) mg = FLT_MAX;
                }
            }
            margins[j] = mg;
        }
        prev = tokens[j];
    }
    free(z);
    return OR_OK;
}

/* =========================================================================
 * Vocabulary-sharded emulator ("PP1 q transport and scheduling design",
 * Sparse support and vocabulary-sharded TP2 follow-up): the vocabulary is
 * split into n_sh contiguous shards [s*Vs, min(V, (s+1)*Vs)), Vs =
 * ceil(V / n_sh), and every step that needs the whole row is an explicit
 * exchange of per-shard partials:
 *   - dense q: all-reduce max, all-reduce the uint64 weight sums and the
 *     floor sums, then the remaining tickets granted globally: each shard
 *     offers its own R best remainders (remainder desc, id asc), the leader
 *     merges them and the R best win;
 *   - top-k q: each shard's local top-k (y desc, id asc), the leader merges
 *     the at most n_sh * k candidates into the global top-k and allocates on
 *     that support;
 *   - draw: the leader's one 24-bit draw selects the shard by the shards'
 *     count totals, and the shard picks the token inside;
 *   - ratio verification: all-reduce of (max, shifted sum) for p, p(x) from
 *     the shard owning x, the test at the leader; the residual draw selects
 *     the shard by the shards' residual masses, then the token inside.
 * Its integer outputs equal those of the unsharded functions (the tests pin
 * that); only p's rounding order differs.
 * ========================================================================= */
typedef struct { double r; int32_t id; } or_rem;

static int or_rem_before(const or_rem* a, const or_rem* b)
{
    return a->r > b->r || (a->r == b->r && a->id < b->id);
}

static int or_cmp_rem_sh(const void* a, const void* b)
{
    const or_rem* u = (const or_rem*)a;
    const or_rem* v = (const or_rem*)b;
    return or_rem_before(u, v) ? -1 : (or_rem_before(v, u) ? 1 : 0);
}

/* One draft row, dense (top_k == 0) or top-k, counts into dense[V]. */
int oracle_q_build_row_sharded(const float* x, int32_t V, float T, int32_t top_k,
                               int32_t n_sh, uint32_t* dense)
{
    memset(dense, 0, sizeof(uint32_t) * (size_t)V);
    if (!(isfinite(T) && T > 0.0f)) return OR_BAD_TEMPERATURE;
    float invT = 1.0f / T;
    if (!(isfinite(invT) && invT >= 0x1p-126f)) return OR_BAD_TEMPERATURE;
    const int32_t Vs = (V + n_sh - 1) / n_sh;
    float* y = (float*)malloc(sizeof(float) * (size_t)V);
    uint8_t* sup = (uint8_t*)calloc((size_t)V, 1);
    if (!y || !sup) { free(y); free(sup); return -1; }
    int st = OR_OK;
    /* per shard: validate and scale; then the all-reduce of "any finite" */
    int32_t n_finite = 0;
    for (int32_t s = 0; s < n_sh && st == OR_OK; ++s) {
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
            float xv = x[v];
            if (isnan(xv) || xv == INFINITY) { st = OR_NONFINITE; break; }
            y[v] = xv * invT;
            if (isfinite(xv) && !isfinite(y[v])) { st = OR_NONFINITE; break; }
            if (y[v] > -INFINITY) ++n_finite;
        }
    }
    if (st == OR_OK && n_finite == 0) st = OR_ZERO_MASS;
    if (st != OR_OK) { free(y); free(sup); return st; }

    /* support: all finite (dense), or the merge of the shards' local top-k */
    if (top_k > 0 && top_k < n_finite) {
        or_yid* cand = (or_yid*)malloc(sizeof(or_yid) * (size_t)(n_sh * top_k + 1));
        or_yid* loc = (or_yid*)malloc(sizeof(or_yid) * (size_t)(Vs + 1));
        int32_t nc = 0;
        for (int32_t s = 0; s < n_sh; ++s) {
            int32_t nl = 0;
            for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v)
                if (y[v] > -INFINITY) { loc[nl].y = y[v]; loc[nl].id = v; ++nl; }
            qsort(loc, (size_t)nl, sizeof(or_yid), or_cmp_topk);
            for (int32_t i = 0; i < nl && i < top_k; ++i) cand[nc++] = loc[i];
        }
        qsort(cand, (size_t)nc, sizeof(or_yid), or_cmp_topk);       /* leader merge */
        for (int32_t i = 0; i < top_k; ++i) sup[cand[i].id] = 1;
        free(cand);
        free(loc);
    } else {
        for (int32_t v = 0; v < V; ++v) sup[v] = (y[v] > -INFINITY);
    }
    /* all-reduce max over the support */
    float m = -INFINITY;
    for (int32_t s = 0; s < n_sh; ++s) {
        float ms = -INFINITY;
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) if (sup[v] && y[v] > ms) ms = y[v];
        if (ms > m) m = ms;
    }
    /* per shard E and uint64 sums; all-reduce */
    uint64_t* E = (uint64_t*)calloc((size_t)V, sizeof(uint64_t));
    uint64_t S = 0;
    for (int32_t s = 0; s < n_sh; ++s) {
        uint64_t Ss = 0;
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
            if (!sup[v]) continue;
            float e = oracle_exp_ds(y[v] - m);
            E[v] = (uint64_t)floor((double)e * 1099511627776.0);
            Ss += E[v];
        }
        S += Ss;
    }
    /* floors per shard, all-reduce F; then the global remaining-ticket grant */
    double k = 16777216.0 / (double)S;
    uint64_t F = 0;
    int32_t npos = 0;
    double* r = (double*)calloc((size_t)V, sizeof(double));
    for (int32_t v = 0; v < V; ++v) {
        if (!sup[v]) continue;
        double a = (double)E[v] * k;
        double f = floor(a);
        dense[v] = (uint32_t)f;
        r[v] = a - f;
        F += (uint64_t)f;
        if (r[v] > 0.0) ++npos;
    }
    if (F > (uint64_t)OR_M || (uint64_t)OR_M - F >= (uint64_t)OR_M ||
        (uint64_t)OR_M - F > (uint64_t)npos) {
        st = OR_ALLOC_INCONSISTENT;
    } else {
        const int64_t R = (int64_t)OR_M - (int64_t)F;
        or_rem* offers = (or_rem*)malloc(sizeof(or_rem) * (size_t)(n_sh * (R + 1) + 1));
        or_rem* loc = (or_rem*)malloc(sizeof(or_rem) * (size_t)(Vs + 1));
        int64_t no = 0;
        for (int32_t s = 0; s < n_sh; ++s) {
            int32_t nl = 0;
            for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v)
                if (sup[v]) { loc[nl].r = r[v]; loc[nl].id = v; ++nl; }
            qsort(loc, (size_t)nl, sizeof(or_rem), or_cmp_rem_sh);
            for (int64_t i = 0; i < nl && i < R; ++i) offers[no++] = loc[i];
        }
        qsort(offers, (size_t)no, sizeof(or_rem), or_cmp_rem_sh);
        for (int64_t i = 0; i < R; ++i) dense[offers[i].id] += 1u;
        free(offers);
        free(loc);
        uint64_t total = 0;
        for (int32_t v = 0; v < V; ++v) total += dense[v];
        if (total != (uint64_t)OR_M) st = OR_ALLOC_INCONSISTENT;
    }
    if (st != OR_OK) memset(dense, 0, sizeof(uint32_t) * (size_t)V);
    free(y); free(sup); free(E); free(r);
    return st;
}

/* The draw over dense counts: the shard by the shards' count totals, then the
 * token inside it. */
int32_t oracle_draw_sharded(const uint32_t* counts, int32_t V, int32_t n_sh, uint32_t D)
{
    const int32_t Vs = (V + n_sh - 1) / n_sh;
    uint64_t before = 0;
    for (int32_t s = 0; s < n_sh; ++s) {
        uint64_t Cs = 0;
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) Cs += counts[v];
        if ((uint64_t)D < before + Cs) {
            uint64_t cum = before;
            for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
                cum += counts[v];
                if (cum > (uint64_t)D) return v;
            }
        }
        before += Cs;
    }
    return -1;
}

/* Target p of one row from the shards' (max, shifted sum) partials. */
static int or_target_row_sharded(const float* z, int32_t V, int32_t n_sh, double* p)
{
    const int32_t Vs = (V + n_sh - 1) / n_sh;
    double M = -INFINITY;
    double* ms = (double*)malloc(sizeof(double) * (size_t)n_sh * 2);
    double* ss = ms + n_sh;
    for (int32_t s = 0; s < n_sh; ++s) {
        float m = -INFINITY;
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
            if (isnan(z[v]) || z[v] == INFINITY) { free(ms); return OR_NONFINITE; }
            if (z[v] > m) m = z[v];
        }
        double sum = 0.0;
        for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v)
            if (z[v] > -INFINITY) sum += exp((double)z[v] - (double)m);
        ms[s] = m;
        ss[s] = sum;
        if (m > M) M = m;
    }
    if (M == -INFINITY) { free(ms); return OR_ZERO_MASS; }
    double Z = 0.0;
    for (int32_t s = 0; s < n_sh; ++s)
        if (ms[s] > -INFINITY) Z += ss[s] * exp(ms[s] - M);
    for (int32_t v = 0; v < V; ++v)
        p[v] = (z[v] == -INFINITY) ? 0.0 : exp((double)z[v] - M) / Z;
    free(ms);
    return OR_OK;
}

/* Residual (or bonus) draw: the shard by the shards' residual masses, then the
 * token inside; flags as in oracle_residual_pick. */
static int32_t or_residual_pick_sharded(const double* p, const uint32_t* c, int32_t V,
                                        int32_t n_sh, uint32_t w, uint32_t* flags)
{
    const int32_t Vs = (V + n_sh - 1) / n_sh;
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* Zs = (double*)calloc((size_t)n_sh, sizeof(double));
    double Z = 0.0;
    int degenerate = 0;
    for (int pass = 0; pass < 2; ++pass) {
        Z = 0.0;
        for (int32_t s = 0; s < n_sh; ++s) {
            Zs[s] = 0.0;
            for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
                double q = (c && !degenerate) ? (double)c[v] / 16777216.0 : 0.0;
                double rv = p[v] - q;
                r[v] = rv > 0.0 ? rv : 0.0;
                Zs[s] += r[v];
            }
            Z += Zs[s];
        }
        if (Z > 0.0 || !c || degenerate) break;
        degenerate = 1;
        if (flags) *flags |= OR_FLAG_DEGENERATE;
    }
    double t = ((double)w * 0x1p-32) * Z;
    int32_t pick = -1, last_pos = -1;
    double before = 0.0, cum = 0.0, prev = 0.0;
    for (int32_t s = 0; s < n_sh && pick < 0; ++s) {
        if (t < before + Zs[s] || s == n_sh - 1) {
            cum = before;
            for (int32_t v = s * Vs; v < V && v < (s + 1) * Vs; ++v) {
                if (r[v] > 0.0) last_pos = v;
                prev = cum;
                cum += r[v];
                if (cum > t) { pick = v; break; }
            }
        }
        before += Zs[s];
    }
    if (pick < 0) {
        for (int32_t v = V - 1; v >= 0; --v) if (r[v] > 0.0) { last_pos = v; break; }
        pick = last_pos;
        prev = cum - (last_pos >= 0 ? r[last_pos] : 0.0);
    }
    if (flags && (fabs(t - prev) <= 1e-6 || fabs(cum - t) <= 1e-6))
        *flags |= OR_FLAG_NEAR_BOUNDARY;
    if (flags && pick >= 0 &&
        (fabs(t - prev) <= 1e-6 * r[pick] || fabs(cum - t) <= 1e-6 * r[pick]))
        *flags |= OR_FLAG_NEAR_BOUNDARY_REL;
    free(r);
    free(Zs);
    return pick;
}

/* Ratio verification of one request with dense q, sharded. */
int oracle_verify_ratio_req_sharded(const float* z, int64_t ld, int32_t V, int32_t depth,
                                    const int32_t* drafts, const uint32_t* counts,
                                    int32_t n_sh, uint64_t seed, uint32_t request,
                                    int32_t* accept_len, int32_t* committed, uint32_t* flags)
{
    uint32_t fl = 0;
    or_discard(depth, accept_len, committed);
    if (flags) *flags = 0;
    for (int32_t j = 0; j < depth; ++j)
        if (drafts[j] < 0 || drafts[j] >= V) return OR_BAD_DRAFT;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    int st = OR_OK;
    int32_t L = depth, pick = -1;
    for (int32_t j = 0; j < depth; ++j) {
        st = or_target_row_sharded(z + (int64_t)j * ld, V, n_sh, p);
        if (st != OR_OK) goto done;
        const uint32_t* q = counts + (int64_t)j * V;
        uint32_t c = q[drafts[j]];
        if (c == 0) { st = OR_BAD_DRAFT; goto done; }
        uint32_t U = oracle_draw_u32(seed, request, (uint32_t)j, OR_PURPOSE_ACCEPT) >> 8;
        double pj = p[drafts[j]];
        double uq = (double)((uint64_t)U * (uint64_t)c) * 0x1p-48;
        if (fabs(uq - pj) <= 1e-6 * ((double)c * 0x1p-24)) fl |= OR_FLAG_AMBIG_ACCEPT;
        if (!oracle_ratio_accept(U, c, pj)) {
            L = j;
            uint64_t total = 0;
            for (int32_t v = 0; v < V; ++v) total += q[v];
            if (total != (uint64_t)OR_M) { st = OR_BAD_Q; goto done; }
            uint32_t w = oracle_draw_u32(seed, request, (uint32_t)j, OR_PURPOSE_RESIDUAL);
            pick = or_residual_pick_sharded(p, q, V, n_sh, w, &fl);
            break;
        }
    }
    if (L == depth) {
        st = or_target_row_sharded(z + (int64_t)depth * ld, V, n_sh, p);
        if (st != OR_OK) goto done;
        uint32_t w = oracle_draw_u32(seed, request, (uint32_t)depth, OR_PURPOSE_BONUS);
        pick = or_residual_pick_sharded(p, NULL, V, n_sh, w, &fl);
    }
    *accept_len = L;
    for (int32_t i = 0; i < L; ++i) committed[i] = drafts[i];
    committed[L] = pick;
done:
    if (st != OR_OK) { or_discard(depth, accept_len, committed); fl = 0; }
    if (flags) *flags = fl;
    free(p);
    return st;
}
