/*
 * tps_oracle.c -- float64 CPU oracle for the batched sampler chain
 *                 temperature -> min-p -> top-k -> top-p -> renormalise -> sample.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no source, header, table or helper
 * with the CUDA library; the two meet only through the seeded synthetic inputs.
 *
 * Plain, slow and literal on purpose: every row is sorted, grouped into classes of equal logits
 * and walked once, all in float64.  Sources, by page title:
 *   [NS]  "Top-p (Nucleus) Sampling, in depth"                                  (aicassindra.com)
 *   [TRT] "Top-p (Nucleus) Sampling"                           (TensorRT-Model-Connect features)
 *   [IMP] "Implement batched top-p sampling with temperature"                (inferenceinterviews)
 *   [ORD] "What do temperature, top-k and top-p each do to the next-token distribution, and in
 *          what order does a serving engine apply them?"                      (inferenceinterviews)
 *
 * Readings where the pages are silent or disagree (each is listed again in the design notes):
 *   - chain order temperature -> min-p -> top-k -> top-p -> sample ([ORD] TL;DR);
 *   - top-p keeps token i iff the mass of strictly more probable tokens is below p ([IMP] "How to
 *     approach it"); "more probable" is decided on the logits, which order exactly like the exact
 *     probabilities for T > 0, so tied logits share a fate;
 *   - that mass is measured after min-p and top-k, renormalised over their survivors S
 *     ([ORD] "A strong answer": the reference sampler recomputes the softmax after the masks);
 *   - T <= 0 is greedy with the lowest index winning ties ([IMP] "A strong answer", item 4);
 *   - p >= 1 keeps S; p <= 0 keeps only the class of the maximum logit (the argmax is always kept,
 *     [NS] "Boundaries and ties");
 *   - min-p keeps p_i >= min_p * p_max ([IMP] "What interviewers probe next"); min_p is clamped
 *     to at most 1; top-k keeps z_i >= the k-th largest logit, ties included, and is off for
 *     k <= 0 or k >= V ([ORD] reference sampler);
 *   - NaN or +inf logits fail the row ([NS] "Failure modes"); a row with no finite logit and a
 *     non-finite T, p or min_p also fail it; -inf logits get probability 0 ([IMP] item 5);
 *   - the draw is an exponential race, argmax P_i / E_i with E_i = -ln u_i ([ORD] "A strong
 *     answer", last paragraph), taken as argmax of  -(zmax - z_i)/T - ln(-ln u_i)  (the row
 *     constant ln Z is dropped), lowest index on equal keys;
 *   - u_i comes from Philox4x32-10 keyed by the row's 64-bit seed, counter
 *     (floor(i/4), row, step_lo, step_hi), word i mod 4, mapped to (2*(x>>9)+1) * 2^-24.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TPSO_ROW_OK 0
#define TPSO_ROW_NAN 1
#define TPSO_ROW_ALL_MASKED 2
#define TPSO_ROW_BAD_PARAM 3

/* Flags describing rows where a floating-point decision sits on a knife edge. */
#define TPSO_FLAG_TOPP_BAND 1 /* normalised mass above some class of S within TOPP_BAND of p     */
#define TPSO_FLAG_MINP_BAND 2 /* some e_i within MINP_BAND (relative) of min_p                   */
#define TPSO_FLAG_RACE_BAND 4 /* best and second-best race keys within RACE_BAND (relative)     */

static const double TOPP_BAND = 1e-6;
static const double MINP_BAND = 1e-12;
static const double RACE_BAND = 1e-12;

/* ---------------------------------------------------------------------------------------------
 * Philox4x32-10, written from its published definition (Salmon, Moraes, Dror, Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
 * round constants below, the key bumped by the two Weyl constants between rounds.
 * ------------------------------------------------------------------------------------------- */
static const uint32_t PHILOX_M0 = 0xD2511F53u;
static const uint32_t PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u;
static const uint32_t PHILOX_W1 = 0xBB67AE85u;

void tpso_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform the race uses for token `token` of row `row` at step `step`. */
double tpso_uniform(uint64_t seed, uint64_t row, uint64_t step, uint64_t token)
{
    uint32_t ctr[4] = {(uint32_t)(token / 4u), (uint32_t)row, (uint32_t)step, (uint32_t)(step >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    tpso_philox4x32_10(ctr, key, x);
    uint32_t w = x[token % 4u];
    return ((double)(2u * (w >> 9) + 1u)) * 0x1p-24;
}

/* The uniform of token `token` in round `round` of the rejection draw: the same generator and
 * mapping, with round + 1 in bits 18..31 of the counter's first word (token / 4 < 2^18 for
 * V <= 2^20), so no round's uniforms coincide with the select path's (which has 0 there). */
double tpso_uniform_round(uint64_t seed, uint64_t row, uint64_t step, uint64_t token, uint32_t round)
{
    uint32_t ctr[4] = {(uint32_t)(token / 4u) | ((round + 1u) << 18), (uint32_t)row, (uint32_t)step,
                       (uint32_t)(step >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    tpso_philox4x32_10(ctr, key, x);
    uint32_t w = x[token % 4u];
    return ((double)(2u * (w >> 9) + 1u)) * 0x1p-24;
}

/* The uniforms of speculative acceptance: the same generator and mapping with bit 31 of the counter's
 * row word set.  Row indices stay below 2^31, so neither the race nor any rejection round uses these
 * counters.  Token TPSO_SPEC_ACCEPT_SLOT (2^20 - 1, above every token index) gives the acceptance
 * test's uniform; a token index gives that token's uniform in the residual race. */
#define TPSO_SPEC_ACCEPT_SLOT 0xFFFFFu
double tpso_uniform_spec(uint64_t seed, uint64_t row, uint64_t step, uint64_t token)
{
    uint32_t ctr[4] = {(uint32_t)(token / 4u), (uint32_t)row | 0x80000000u, (uint32_t)step, (uint32_t)(step >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    tpso_philox4x32_10(ctr, key, x);
    uint32_t w = x[token % 4u];
    return ((double)(2u * (w >> 9) + 1u)) * 0x1p-24;
}

/* Race key of a kept token: ln P_i - ln E_i up to the row constant ln Z. */
static double race_key(double zmax, double zi, double T, double u)
{
    double d = (zmax - zi) / T;
    return -d - log(-log(u));
}

/* Sort order: logit descending, then index ascending (so the walk is deterministic). */
typedef struct {
    double z;
    int64_t i;
} zi_pair;

static int cmp_desc(const void* a, const void* b)
{
    const zi_pair* x = (const zi_pair*)a;
    const zi_pair* y = (const zi_pair*)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

typedef struct {
    int32_t token, status, kept, flags;
    double cutoff, z_s, z_k, n_s;
} row_out;

/* One row, straight from the definition.  `pairs` and `e` are scratch of length V. */
static void sample_row(const double* z, int64_t V, double T, int32_t k, double p, double m,
                       uint64_t seed, uint64_t row_id, uint64_t step, double* probs,
                       zi_pair* pairs, double* e, row_out* r, int draw, int32_t* rounds)
{
    if (rounds) *rounds = 0;
    memset(r, 0, sizeof(*r));
    r->token = -1;
    r->cutoff = NAN;
    if (probs)
        for (int64_t i = 0; i < V; ++i) probs[i] = 0.0;

    /* Validate ([NS] "Failure modes": NaN fails the request; +inf is treated the same way). */
    double zmax = -INFINITY;
    int64_t n_finite = 0;
    for (int64_t i = 0; i < V; ++i) {
        double v = z[i];
        if (isnan(v) || v == INFINITY) {
            r->status = TPSO_ROW_NAN;
            return;
        }
        if (v > -INFINITY) {
            ++n_finite;
            if (v > zmax) zmax = v;
        }
    }
    if (!isfinite(T) || !isfinite(p) || !isfinite(m)) {
        r->status = TPSO_ROW_BAD_PARAM;
        return;
    }
    if (n_finite == 0) {
        r->status = TPSO_ROW_ALL_MASKED;
        return;
    }

    /* Greedy branch: T <= 0 takes the argmax, lowest index on ties ([IMP] "A strong answer"). */
    if (T <= 0.0) {
        int64_t arg = -1;
        for (int64_t i = 0; i < V; ++i)
            if (z[i] == zmax) { arg = i; break; }
        r->token = (int32_t)arg;
        r->kept = 1;
        r->cutoff = zmax;
        r->z_s = r->z_k = r->n_s = 1.0;
        if (probs) probs[arg] = 1.0;
        return;
    }

    /* Tempered ratios e_i = exp(z_i/T) / exp(zmax/T) ([ORD] the p_i(T) equation; [IMP] item 1:
     * the max is subtracted before exp); -inf logits get 0 ([IMP] item 5). */
    int64_t n = 0;
    for (int64_t i = 0; i < V; ++i) {
        if (z[i] > -INFINITY) {
            e[i] = exp(-((zmax - z[i]) / T));
            pairs[n].z = z[i];
            pairs[n].i = i;
            ++n;
        } else {
            e[i] = 0.0;
        }
    }
    qsort(pairs, (size_t)n, sizeof(zi_pair), cmp_desc);

    /* min-p: keep p_i >= min_p * p_max, i.e. e_i >= min_p ([IMP] probe on min-p; [ORD]). */
    double mm = m > 1.0 ? 1.0 : m;
    /* top-k: keep z_i >= the k-th largest finite logit, ties included ([ORD] reference sampler). */
    double vk = -INFINITY;
    if (k > 0 && (int64_t)k < V && (int64_t)k < n) vk = pairs[k - 1].z;

    /* S = survivors of both masks.  Both are upper sets in z, so S is a prefix of the order. */
    int64_t ns = 0;
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = pairs[t].i;
        int in_minp = (mm > 0.0) ? (e[i] >= mm) : 1;
        if (mm > 0.0 && fabs(e[i] - mm) <= MINP_BAND * mm) r->flags |= TPSO_FLAG_MINP_BAND;
        int in_topk = pairs[t].z >= vk;
        if (in_minp && in_topk) {
            if (ns != t) abort(); /* survivors must form a prefix of the sorted order */
            ++ns;
        }
    }
    /* ns >= 1: the maximum has e = 1 >= min(m,1) and is >= the k-th largest. */
    double zs = 0.0;
    for (int64_t t = 0; t < ns; ++t) zs += e[pairs[t].i];

    /* top-p over S, class by class ([IMP] "How to approach it": keep i iff the mass of strictly
     * more probable tokens is below p; tied tokens share that mass and so share a fate).  The
     * class of the maximum is always kept ([NS] "Boundaries and ties": never empty). */
    int64_t nk = ns;
    if (p < 1.0) {
        double above = 0.0;
        int64_t t = 0;
        int first = 1;
        nk = 0;
        while (t < ns) {
            int64_t u = t;
            double cls = 0.0;
            while (u < ns && pairs[u].z == pairs[t].z) {
                cls += e[pairs[u].i];
                ++u;
            }
            if (!first && fabs(above / zs - p) < TOPP_BAND) r->flags |= TPSO_FLAG_TOPP_BAND;
            if (first || above < p * zs) {
                nk = u;
            } else {
                /* classes further down have even more mass above them; keep scanning only for
                 * the band flag */
            }
            above += cls;
            first = 0;
            t = u;
        }
    }

    /* Renormalise once, at the end ([IMP] "What interviewers probe next"; [ORD] mistakes). */
    double zk = 0.0;
    for (int64_t t = 0; t < nk; ++t) zk += e[pairs[t].i];
    if (probs)
        for (int64_t t = 0; t < nk; ++t) probs[pairs[t].i] = e[pairs[t].i] / zk;

    r->kept = (int32_t)nk;
    r->cutoff = pairs[nk - 1].z;
    r->z_s = zs;
    r->z_k = zk;
    r->n_s = (double)ns;

    if (draw == 1) {
        /* Sort-free top-p by rejection ([NS] "Sort-free top-p by rejection sampling"): each round
         * races among the survivors above the pivot (all of S at first), in proportion to e_i; the
         * winner t is accepted when the mass of strictly more probable survivors is below p * Z_S
         * -- the same test that defines the kept set, so the class of the maximum always passes --
         * and otherwise t's logit becomes the pivot, dropping t's class and everything below. */
        double zpiv = -INFINITY;
        for (uint32_t round = 0; round < (1u << 16); ++round) {
            double best = -INFINITY;
            int64_t arg = -1;
            for (int64_t t = 0; t < ns; ++t) {
                if (!(pairs[t].z > zpiv)) continue;
                int64_t i = pairs[t].i;
                double key = race_key(zmax, z[i], T, tpso_uniform_round(seed, row_id, step, (uint64_t)i, round));
                if (key > best || (key == best && i < arg)) {
                    best = key;
                    arg = i;
                }
            }
            double above = 0.0;
            for (int64_t t = 0; t < ns; ++t)
                if (pairs[t].z > z[arg]) above += e[pairs[t].i];
            if (rounds) *rounds = (int32_t)(round + 1);
            if (z[arg] == zmax || p >= 1.0 || above < p * zs) {
                r->token = (int32_t)arg;
                return;
            }
            zpiv = z[arg];
        }
        r->token = -1; /* unreachable: every rejection removes at least one class */
        return;
    }

    /* Exponential race over the kept set ([ORD] "A strong answer": argmax p / Exp(1)). */
    double best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int64_t t = 0; t < nk; ++t) {
        int64_t i = pairs[t].i;
        double u = tpso_uniform(seed, row_id, step, (uint64_t)i);
        double key = race_key(zmax, z[i], T, u);
        if (key > best || (key == best && i < arg)) {
            second = best;
            best = key;
            arg = i;
        } else if (key > second) {
            second = key;
        }
    }
    if (nk > 1 && best - second <= RACE_BAND * fmax(1.0, fabs(best))) r->flags |= TPSO_FLAG_RACE_BAND;

    r->token = (int32_t)arg;
}

/*
 * Batched entry point.  z: [B, ld] float64 (the exact widened fp32/bf16 logits), rows of length V.
 * T, p, m: [B] float64 (the exact widened fp32 parameters); k: [B]; seed: [B]; row_ids: nullable
 * [B] (the row index the Philox counter uses; defaults to b).  Outputs are [B] except
 * out_probs ([B, V], nullable) and out_aux ([B, 3] = Z_S, Z_K, |S|, nullable).
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 when scratch cannot be allocated.
 */
static int sample_batch(const double* z, int64_t B, int64_t V, int64_t ld, const double* T, const int32_t* k,
                        const double* p, const double* m, const uint64_t* seed, const int64_t* row_ids,
                        uint64_t step, int32_t* out_token, double* out_probs, int32_t* out_status,
                        double* out_cutoff, int32_t* out_kept, int32_t* out_flags, double* out_aux,
                        int nthreads, int draw, int32_t* out_rounds)
{
    if (B <= 0) return 0;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        zi_pair* pairs = (zi_pair*)malloc(sizeof(zi_pair) * (size_t)V);
        double* e = (double*)malloc(sizeof(double) * (size_t)V);
        if (!pairs || !e) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t b = 0; b < B; ++b) {
                row_out r;
                uint64_t rid = row_ids ? (uint64_t)row_ids[b] : (uint64_t)b;
                sample_row(z + b * ld, V, T[b], k[b], p[b], m[b], seed[b], rid, step,
                           out_probs ? out_probs + b * V : NULL, pairs, e, &r, draw,
                           out_rounds ? out_rounds + b : NULL);
                out_token[b] = r.token;
                if (out_status) out_status[b] = r.status;
                if (out_cutoff) out_cutoff[b] = r.cutoff;
                if (out_kept) out_kept[b] = r.kept;
                if (out_flags) out_flags[b] = r.flags;
                if (out_aux) {
                    out_aux[3 * b + 0] = r.z_s;
                    out_aux[3 * b + 1] = r.z_k;
                    out_aux[3 * b + 2] = r.n_s;
                }
            }
        }
        free(pairs);
        free(e);
    }
    return failed ? -1 : 0;
}

int tpso_sample(const double* z, int64_t B, int64_t V, int64_t ld, const double* T, const int32_t* k,
                const double* p, const double* m, const uint64_t* seed, const int64_t* row_ids,
                uint64_t step, int32_t* out_token, double* out_probs, int32_t* out_status,
                double* out_cutoff, int32_t* out_kept, int32_t* out_flags, double* out_aux,
                int nthreads)
{
    return sample_batch(z, B, V, ld, T, k, p, m, seed, row_ids, step, out_token, out_probs, out_status, out_cutoff,
                        out_kept, out_flags, out_aux, nthreads, 0, NULL);
}

/* The same rows drawn by rejection rounds instead of one race over the kept set (same kept set,
 * same distribution, different uniforms); out_rounds[b] = rounds row b took. */
int tpso_sample_rejection(const double* z, int64_t B, int64_t V, int64_t ld, const double* T, const int32_t* k,
                          const double* p, const double* m, const uint64_t* seed, const int64_t* row_ids,
                          uint64_t step, int32_t* out_token, double* out_probs, int32_t* out_status,
                          double* out_cutoff, int32_t* out_kept, int32_t* out_flags, double* out_aux,
                          int nthreads, int32_t* out_rounds)
{
    return sample_batch(z, B, V, ld, T, k, p, m, seed, row_ids, step, out_token, out_probs, out_status, out_cutoff,
                        out_kept, out_flags, out_aux, nthreads, 1, out_rounds);
}

int tpso_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------------------------
 * Speculative acceptance on truncated distributions ([NS] "Logprobs, speculative decoding and
 * reproducibility": accept a draft token x with probability min(1, P(x)/Q(x)); on rejection draw
 * from the normalised positive part of P - Q; P is the target's truncated and renormalised
 * distribution, Q the distribution the draft actually sampled from, truncation included).
 *   P = the renormalised kept distribution of the target row under its (T, k, p, m) -- exactly the
 *       probability row the chain above produces (one-hot for a greedy target);
 *   Q = the same for the draft row under the draft's (T, k, p, m);
 *   accepted iff u * Q(x) < P(x), with u the acceptance uniform (an odd multiple of 2^-24 in (0, 1),
 *       so this holds with probability min(1, P(x)/Q(x)) up to the 2^-23 grid);
 *   otherwise the token is argmax over i with r_i = P_i - Q_i > 0 of ln r_i - ln(-ln u_i) (an
 *       exponential race over the residual; lowest index on equal keys).  With exact arithmetic a
 *       rejection leaves some r_i > 0 (P and Q both sum to 1 and P(x) < Q(x)); if rounding leaves
 *       none, P and Q agree, and since P = Q accepts every draft, x stands (accepted).
 * A row fails (token -1, not accepted) when the target or the draft row fails, or when x is not a
 * token the draft distribution can produce (outside [0, V), or Q(x) = 0): TPSO_ROW_BAD_PARAM.
 * Flags: the target's top-p / min-p band flags in bits 0-1, the draft's in bits 4-5; bit 3 when
 * u Q(x) and P(x) lie within SPEC_BAND (relative) of each other; bit 2 when the two best residual
 * race keys lie within the error the residuals' rounding allows.
 * --------------------------------------------------------------------------------------------- */
#define TPSO_FLAG_ACCEPT_BAND 8
static const double SPEC_BAND = 1e-5;

int tpso_spec_accept(const double* zt, const double* zd, int64_t B, int64_t V, int64_t ld, const double* Tt,
                     const int32_t* kt, const double* pt, const double* mt, const double* Td, const int32_t* kd,
                     const double* pd, const double* md, const int32_t* draft, const uint64_t* seed,
                     const int64_t* row_ids, uint64_t step, int32_t* out_token, int32_t* out_accepted,
                     int32_t* out_status, int32_t* out_flags, double* out_px, double* out_qx, int nthreads)
{
    if (B <= 0) return 0;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        zi_pair* pairs = (zi_pair*)malloc(sizeof(zi_pair) * (size_t)V);
        double* e = (double*)malloc(sizeof(double) * (size_t)V);
        double* P = (double*)malloc(sizeof(double) * (size_t)V);
        double* Q = (double*)malloc(sizeof(double) * (size_t)V);
        if (!pairs || !e || !P || !Q) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t b = 0; b < B; ++b) {
                uint64_t rid = row_ids ? (uint64_t)row_ids[b] : (uint64_t)b;
                row_out rt, rd;
                sample_row(zt + b * ld, V, Tt[b], kt[b], pt[b], mt[b], seed[b], rid, step, P, pairs, e, &rt, 0, NULL);
                sample_row(zd + b * ld, V, Td[b], kd[b], pd[b], md[b], seed[b], rid, step, Q, pairs, e, &rd, 0, NULL);
                int32_t x = draft[b];
                int32_t status = rt.status != TPSO_ROW_OK ? rt.status : rd.status;
                if (status == TPSO_ROW_OK && (x < 0 || (int64_t)x >= V || !(Q[x] > 0.0))) status = TPSO_ROW_BAD_PARAM;
                int32_t flags = (rt.flags & 3) | ((rd.flags & 3) << 4);
                int32_t token = -1, accepted = 0;
                double px = NAN, qx = NAN;
                if (status == TPSO_ROW_OK) {
                    px = P[x];
                    qx = Q[x];
                    double u = tpso_uniform_spec(seed[b], rid, step, TPSO_SPEC_ACCEPT_SLOT);
                    double lhs = u * qx;
                    if (fabs(lhs - px) <= SPEC_BAND * fmax(lhs, px)) flags |= TPSO_FLAG_ACCEPT_BAND;
                    if (lhs < px) {
                        accepted = 1;
                        token = x;
                    } else {
                        double best = -INFINITY, second = -INFINITY, tol_best = 0.0, tol_second = 0.0;
                        for (int64_t i = 0; i < V; ++i) {
                            double r = P[i] - Q[i];
                            if (!(r > 0.0)) continue;
                            double key = log(r) - log(-log(tpso_uniform_spec(seed[b], rid, step, (uint64_t)i)));
                            double tol = SPEC_BAND * (P[i] + Q[i]) / r;
                            if (key > best) {
                                second = best;
                                tol_second = tol_best;
                                best = key;
                                tol_best = tol;
                                token = (int32_t)i;
                            } else if (key > second) {
                                second = key;
                                tol_second = tol;
                            }
                        }
                        if (second > -INFINITY && best - second <= tol_best + tol_second + 1e-12) flags |= TPSO_FLAG_RACE_BAND;
                        if (token < 0) {  /* no P_i above Q_i after rounding: P = Q, and x stands */
                            token = x;
                            accepted = 1;
                        }
                    }
                }
                out_token[b] = token;
                if (out_accepted) out_accepted[b] = accepted;
                if (out_status) out_status[b] = status;
                if (out_flags) out_flags[b] = flags;
                if (out_px) out_px[b] = px;
                if (out_qx) out_qx[b] = qx;
            }
        }
        free(pairs);
        free(e);
        free(P);
        free(Q);
    }
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------------------------
 * Penalties on the raw logits, ahead of the chain above.  [NS] "Where top-p sits in the sampler
 * chain" puts repetition, frequency and presence penalties first, on the logits; [ORD] "What
 * interviewers probe next" says they act before temperature, on raw logits, so that they change
 * the greedy choice too.  The pages give no formulas; this takes the common ones:
 *   c_t  = number of entries of the row's history equal to t (entries outside [0, V) and past the
 *          row's history length are ignored; the length is clamped to [0, H]);
 *   for every t with c_t > 0:
 *     y   = z_t / r   if z_t > 0,   z_t * r   otherwise          (repetition, r > 0; 1 = off)
 *     z'_t = y - (f * c_t + rho)                                  (frequency f, presence rho)
 *   every other logit is unchanged.
 * Precision: the pages fix none.  The penalised logit is the sampler's input, so it is defined in
 * float32, one correctly rounded operation at a time in the order written, and rounded to
 * bfloat16 (nearest, ties to even) for bfloat16 logits; this oracle performs exactly those float
 * operations (the build disables contraction).  A row with r <= 0 or a non-finite r, f or rho is
 * left unchanged and reported as a bad parameter.
 * --------------------------------------------------------------------------------------------- */

/* Round a float32 to the nearest bfloat16 (ties to even), returned as the float it represents. */
static float round_bf16(float x)
{
    if (isnan(x)) return x;
    uint32_t u;
    memcpy(&u, &x, 4);
    const uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    uint32_t r = keep;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1u;  /* carries into the exponent */
    r <<= 16;
    float y;
    memcpy(&y, &r, 4);
    return y;
}

int tpso_penalties(float* z, int is_bf16, int64_t B, int64_t V, int64_t ld, const int32_t* hist, int64_t H,
                   int64_t ldh, const int32_t* hist_len, const float* rep, const float* freq, const float* pres,
                   int32_t* status)
{
    int32_t* cnt = (int32_t*)calloc((size_t)(V > 0 ? V : 1), sizeof(int32_t));
    if (!cnt) return 1;
    for (int64_t b = 0; b < B; ++b) {
        const float r = rep ? rep[b] : 1.0f;
        const float f = freq ? freq[b] : 0.0f;
        const float rho = pres ? pres[b] : 0.0f;
        if (!(isfinite(r) && r > 0.0f && isfinite(f) && isfinite(rho))) {
            if (status) status[b] = TPSO_ROW_BAD_PARAM;
            continue;
        }
        if (status) status[b] = TPSO_ROW_OK;
        int64_t n = hist_len ? (int64_t)hist_len[b] : H;
        if (n < 0) n = 0;
        if (n > H) n = H;
        memset(cnt, 0, (size_t)V * sizeof(int32_t));
        for (int64_t j = 0; j < n; ++j) {
            const int32_t t = hist[b * ldh + j];
            if (t >= 0 && (int64_t)t < V) ++cnt[t];
        }
        float* row = z + b * ld;
        for (int64_t t = 0; t < V; ++t) {
            if (cnt[t] == 0) continue;
            const float x = row[t];
            const float y = (x > 0.0f) ? x / r : x * r;
            const float s = f * (float)cnt[t] + rho;
            const float out = y - s;
            row[t] = is_bf16 ? round_bf16(out) : out;
        }
    }
    free(cnt);
    return 0;
}
