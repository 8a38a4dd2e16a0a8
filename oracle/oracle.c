/*
 * Plain fp64 CPU oracle for batched speculative-decoding verification and
 * the Adaptive-Verification (AV) acceptance estimator.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * constant or helper with the CUDA library; both sides are written from the
 * pages' description of the method.  Every step is the slow, obvious one:
 * single thread, fp64 arithmetic, ascending vocabulary order.
 *
 * Sources (page title, then section):
 *  [SD]  "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet -- section
 *        "one speculative step" (draft, verify, accept with min(1, ratio),
 *        resample the normalised positive residual at the first rejection,
 *        bonus token when all drafts pass) and the Python loop printed under
 *        "algorithm loop in code" (u < min(1, ratio), ratio = inf when the
 *        drafter's probability is zero).  The cheatsheet names the DRAFT
 *        distribution p and the VERIFIER q; this file uses the AV article's
 *        names instead: p = target (verifier), q = draft.
 *  [AV]  "Adaptive Verification without a confidence head" (and its German
 *        translation "Adaptive Verification ohne Confidence Head") --
 *        "Solution", "Scoring the distribution" (per-position logistic
 *        regression sigmoid(omega * logit(q_max) + beta_i)), "Other features
 *        considered" (survival = cumulative product of confidences),
 *        "Fitting the coefficients" (labels up to and including the first
 *        rejection; IRLS / Newton step H * delta = g with H of size
 *        (K+1)x(K+1); accumulation over a round of N decode steps; shared
 *        slope; damping n / (n + constant)), footnote 1 (two-token example).
 *  [PX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *        1, 2, 3" (SC'11) -- the Philox4x32-10 block function.
 *
 * Readings where the pages are silent:
 *  - temperature tau divides both target and draft logits; tau == 0 is a
 *    greedy row (argmax matching, lowest index on ties, no uniforms drawn);
 *    a greedy row's distributions (for the AV feature) use tau = 1;
 *  - feature x = logit(q_max) = -ln E with E = sum over v != argmax of
 *    exp(y_v - max y) (exactly one copy of the max excluded), clamped to
 *    [-30, 30]; E == 0 gives +30;
 *  - uniform for acceptance at position i: U(seed, b, i, draw 0); for the
 *    residual/bonus draw at position a: U(seed, b, a, draw 1);
 *  - CDF inversion: smallest v (ascending) with C(v) > u * R;
 *  - zero residual mass (only reachable through rounding): sample p instead
 *    and raise flag ORC_FLAG_ZERO_RESIDUAL;
 *  - Newton step: H delta = g (g = gradient of the summed log-loss),
 *    theta <- theta - n/(n + c) * delta; positions without labels keep their
 *    intercept; a ridge 1e-9 * trace(H) / (K+1) is added to the diagonal.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_FLAG_ZERO_RESIDUAL 1
#define ORC_FLAG_NONFINITE 2
#define ORC_FLAG_TOKEN_RANGE 4
#define ORC_FLAG_BAD_LEN 8
#define ORC_FLAG_BAD_TEMP 16

/* ------------------------------------------------------------------------ */
/* [PX] Philox4x32-10.                                                       */
/* One round: two 32x32->64 products of counter words 0 and 2 with the       */
/* round multipliers; the new counter is (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1),    */
/* hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)).  The key is bumped by the Weyl constants */
/* (golden ratio, sqrt(3) - 1) between rounds.  Ten rounds.                  */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    int round;
    for (round = 0; round < 10; round++) {
        uint64_t prod_a, prod_b;
        uint32_t y0, y1, y2, y3;
        if (round > 0) {
            k0 = k0 + 0x9E3779B9u;
            k1 = k1 + 0xBB67AE85u;
        }
        prod_a = (uint64_t)0xD2511F53u * (uint64_t)x0;
        prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        y0 = (uint32_t)(prod_b >> 32) ^ x1 ^ k0;
        y1 = (uint32_t)(prod_b & 0xffffffffu);
        y2 = (uint32_t)(prod_a >> 32) ^ x3 ^ k1;
        y3 = (uint32_t)(prod_a & 0xffffffffu);
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Uniform draw `draw` for sequence b at draft position pos:
 * key = (seed low word, seed high word), counter = (b, pos, draw / 4, 0),
 * output word draw % 4, U = (word >> 8) * 2^-24 in [0, 1 - 2^-24]. */
double orc_uniform(uint64_t seed, uint32_t b, uint32_t pos, uint32_t draw)
{
    uint32_t ctr[4], key[2], out[4];
    ctr[0] = b; ctr[1] = pos; ctr[2] = draw / 4u; ctr[3] = 0u;
    key[0] = (uint32_t)(seed & 0xffffffffu);
    key[1] = (uint32_t)(seed >> 32);
    orc_philox4x32_10(ctr, key, out);
    return (double)(out[draw % 4u] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Logit access: dtype 0 = bf16 (widened exactly), 1 = fp32.                 */
/* ------------------------------------------------------------------------ */
static double logit_at(const void *base, int dtype, size_t idx)
{
    if (dtype == 0) {
        uint16_t h = ((const uint16_t *)base)[idx];
        uint32_t w = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

typedef struct {
    double m;      /* max_v y_v, y = z / tau                     */
    double lnS;    /* ln sum_v exp(y_v - m)                      */
    double E;      /* sum_{v != argmax} exp(y_v - m)             */
    int argmax;    /* lowest index attaining m                   */
    int nonfinite; /* NaN anywhere, or max not finite            */
} orc_row_stats_t;

/* Softmax statistics of one vocabulary row at temperature tau ([SD] "one
 * speculative step": both models return a distribution per position). */
void orc_row_stats(const void *row, int dtype, int V, double tau, orc_row_stats_t *st)
{
    int v;
    double m = -INFINITY, S = 0.0, E = 0.0;
    int arg = 0, bad = 0;
    for (v = 0; v < V; v++) {
        double y = logit_at(row, dtype, (size_t)v) / tau;
        if (isnan(y)) { bad = 1; continue; }
        if (y > m) { m = y; arg = v; }
    }
    if (!isfinite(m)) bad = 1;
    for (v = 0; v < V; v++) {
        double y = logit_at(row, dtype, (size_t)v) / tau;
        double t;
        if (isnan(y)) continue;
        t = exp(y - m);
        S += t;
        if (v != arg) E += t;
    }
    st->m = m;
    st->lnS = log(S);
    st->E = E;
    st->argmax = arg;
    st->nonfinite = bad;
}

/* log p(v) for a row with statistics st. */
static double row_logprob(const void *row, int dtype, double tau, const orc_row_stats_t *st, int v)
{
    return logit_at(row, dtype, (size_t)v) / tau - st->m - st->lnS;
}

/* [AV] "Scoring the distribution": the feature is the log-odds of the
 * drafter's most likely token, logit(q_max) = ln(q_max / (1 - q_max)).
 * With q_max = 1/S and 1 - q_max = E/S this is -ln E. */
double orc_feature(double E)
{
    double x;
    if (E <= 0.0) return 30.0;
    x = -log(E);
    if (x > 30.0) x = 30.0;
    if (x < -30.0) x = -30.0;
    return x;
}

/* [AV] per-position logistic regression: conf = sigmoid(omega * x + beta_i). */
double orc_conf(double omega, double beta, double x)
{
    return 1.0 / (1.0 + exp(-(omega * x + beta)));
}

/* [AV] "Other features considered": survival = cumulative product of the
 * confidences; a draft is kept while its survival is >= the threshold. */
int orc_kept_len(const double *conf, int K, double threshold)
{
    int i, kept = 0;
    double surv = 1.0;
    if (!(threshold > 0.0)) return K;
    for (i = 0; i < K; i++) {
        surv *= conf[i];
        if (surv >= threshold) kept = i + 1;
        else break;
    }
    return kept;
}

/* Draft-only AV scoring: features, confidences, kept lengths. */
void orc_av_score(int B, int K, int V, int dtype, const void *draft, const float *temperature,
                  const double *theta, double keep_threshold,
                  double *out_feature, double *out_conf, int32_t *out_kept_len)
{
    int b, i;
    for (b = 0; b < B; b++) {
        double tau = (double)temperature[b];
        if (!(tau > 0.0)) tau = 1.0;
        for (i = 0; i < K; i++) {
            orc_row_stats_t st;
            const char *row = (const char *)draft + ((size_t)b * K + i) * (size_t)V * (dtype == 0 ? 2 : 4);
            double x;
            orc_row_stats(row, dtype, V, tau, &st);
            x = orc_feature(st.E);
            out_feature[(size_t)b * K + i] = x;
            out_conf[(size_t)b * K + i] = orc_conf(theta[0], theta[1 + i], x);
        }
        out_kept_len[b] = orc_kept_len(out_conf + (size_t)b * K, K, keep_threshold);
    }
}

/* ------------------------------------------------------------------------ */
/* Inverse-CDF draw from a non-negative weight vector r (length V):          */
/* smallest v with C(v) = sum_{w <= v} r_w > u * R.  Returns the token and   */
/* the draw's margin min(C(v) - uR, uR - C(v-1)) / R.                        */
/* ------------------------------------------------------------------------ */
static int cdf_pick(const double *r, int V, double u, double *margin)
{
    int v, tok = -1;
    double R = 0.0, T, C = 0.0, Cprev = 0.0;
    for (v = 0; v < V; v++) R += r[v];
    T = u * R;
    for (v = 0; v < V; v++) {
        Cprev = C;
        C += r[v];
        if (C > T) { tok = v; break; }
    }
    if (tok < 0) { /* cannot happen for R > 0 and u < 1; keep the last positive weight */
        for (v = V - 1; v >= 0; v--) if (r[v] > 0.0) { tok = v; break; }
        *margin = 0.0;
        return tok < 0 ? 0 : tok;
    }
    {
        double a = C - T, b = T - Cprev;
        *margin = (a < b ? a : b) / R;
    }
    return tok;
}

/* ------------------------------------------------------------------------ */
/* One verification step over B sequences ([SD] "one speculative step").    */
/*   target      [B][K+1][V]   draft [B][K][V]   draft_tokens [B][K]         */
/*   draft_len   [B] or NULL (= K): drafts verified for sequence b           */
/*   seq_ids     [B] or NULL: global sequence index used as the uniforms'    */
/*               counter (lets a subset of a batch be checked alone)         */
/*   temperature [B] (0 = greedy)                                            */
/*   theta       [K+1] or NULL: (omega, beta_0..beta_{K-1}); with theta the  */
/*               feature and confidence of every verified draft are written  */
/* Outputs: out_tokens [B][K+1] (-1 padded), out_accept_len [B],             */
/*   out_feature/out_conf [B][K] (NaN where not verified; may be NULL),      */
/*   out_margin [B][2]: smallest acceptance margin |u - ratio| over the     */
/*   acceptance uniforms the sequence consumed, and the sampling margin      */
/*   (distance of u*R to the nearer edge of the chosen CDF step, divided by  */
/*   R); +inf when no such uniform was consumed,                             */
/*   out_ndraws [B]: uniforms consumed, out_flags [B]: ORC_FLAG_* bits.      */
/* ------------------------------------------------------------------------ */
void orc_verify(int B, int K, int V, int dtype,
                const void *target, const void *draft, const int32_t *draft_tokens,
                const int32_t *draft_len, const int32_t *seq_ids, const float *temperature,
                uint64_t seed, const double *theta,
                int32_t *out_tokens, int32_t *out_accept_len,
                double *out_feature, double *out_conf,
                double *out_margin, int32_t *out_ndraws, int32_t *out_flags)
{
    size_t esz = dtype == 0 ? 2 : 4;
    size_t rowb = (size_t)V * esz;
    double *r = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    orc_row_stats_t *tst = (orc_row_stats_t *)malloc(sizeof(orc_row_stats_t) * (size_t)(K + 1));
    orc_row_stats_t *dst = (orc_row_stats_t *)malloc(sizeof(orc_row_stats_t) * (size_t)(K > 0 ? K : 1));
    int b;
    for (b = 0; b < B; b++) {
        double tau = (double)temperature[b];
        int greedy, k, i, j, a, tok, flags = 0, ndraws = 0;
        double margin = INFINITY, smargin = INFINITY;
        const char *trow0 = (const char *)target + (size_t)b * (size_t)(K + 1) * rowb;
        const char *drow0 = (const char *)draft + (size_t)b * (size_t)K * rowb;
        const int32_t *d = draft_tokens + (size_t)b * K;
        uint32_t sid = seq_ids ? (uint32_t)seq_ids[b] : (uint32_t)b;

        if (isnan(tau) || tau < 0.0) { flags |= ORC_FLAG_BAD_TEMP; tau = 0.0; }
        greedy = (tau == 0.0);
        if (greedy) tau = 1.0;

        k = draft_len ? draft_len[b] : K;
        if (k < 0 || k > K) { flags |= ORC_FLAG_BAD_LEN; k = k < 0 ? 0 : K; }

        for (j = 0; j <= k; j++) {
            orc_row_stats(trow0 + (size_t)j * rowb, dtype, V, tau, &tst[j]);
            if (tst[j].nonfinite) flags |= ORC_FLAG_NONFINITE;
        }
        for (i = 0; i < k; i++) {
            orc_row_stats(drow0 + (size_t)i * rowb, dtype, V, tau, &dst[i]);
            if (dst[i].nonfinite) flags |= ORC_FLAG_NONFINITE;
        }
        for (i = 0; i < K; i++) {
            if (out_feature) out_feature[(size_t)b * K + i] = i < k ? orc_feature(dst[i].E) : NAN;
            if (out_conf)
                out_conf[(size_t)b * K + i] =
                    (i < k && theta) ? orc_conf(theta[0], theta[1 + i], orc_feature(dst[i].E)) : NAN;
        }

        /* Left-to-right acceptance; stop at the first rejection. */
        a = k;
        for (i = 0; i < k; i++) {
            int di = d[i];
            int accept;
            int in_range = (di >= 0 && di < V);
            if (!in_range) flags |= ORC_FLAG_TOKEN_RANGE;
            if (greedy) {
                accept = in_range && di == tst[i].argmax;
            } else {
                double u = orc_uniform(seed, sid, (uint32_t)i, 0u);
                double ratio, mg;
                ndraws++;
                if (!in_range) {
                    ratio = 0.0;
                } else {
                    double lp = row_logprob(trow0 + (size_t)i * rowb, dtype, tau, &tst[i], di);
                    double lq = row_logprob(drow0 + (size_t)i * rowb, dtype, tau, &dst[i], di);
                    if (lq == -INFINITY) ratio = INFINITY; /* drafter probability 0 */
                    else ratio = exp(lp - lq);
                }
                mg = fabs(u - ratio);
                if (mg < margin) margin = mg;
                accept = u < ratio; /* u < min(1, ratio) with u in [0, 1) */
            }
            if (!accept) { a = i; break; }
        }

        /* Token at position a: residual (a < k), bonus (a == k), or argmax. */
        if (greedy) {
            tok = tst[a].argmax;
        } else {
            double u2 = orc_uniform(seed, sid, (uint32_t)a, 1u);
            double mg, R = 0.0;
            const char *trow = trow0 + (size_t)a * rowb;
            int v;
            ndraws++;
            if (a < k) {
                const char *drow = drow0 + (size_t)a * rowb;
                for (v = 0; v < V; v++) {
                    double p = exp(row_logprob(trow, dtype, tau, &tst[a], v));
                    double q = exp(row_logprob(drow, dtype, tau, &dst[a], v));
                    double x = p - q;
                    r[v] = x > 0.0 ? x : 0.0;
                    R += r[v];
                }
                if (!(R > 0.0)) flags |= ORC_FLAG_ZERO_RESIDUAL;
            }
            if (a == k || !(R > 0.0)) {
                for (v = 0; v < V; v++) r[v] = exp(row_logprob(trow, dtype, tau, &tst[a], v));
            }
            tok = cdf_pick(r, V, u2, &mg);
            smargin = mg;
        }

        for (j = 0; j <= K; j++) {
            int32_t val = -1;
            if (j < a) val = d[j];
            else if (j == a) val = tok;
            out_tokens[(size_t)b * (K + 1) + j] = val;
        }
        out_accept_len[b] = a;
        if (out_margin) {
            out_margin[2 * (size_t)b] = margin;
            out_margin[2 * (size_t)b + 1] = smargin;
        }
        if (out_ndraws) out_ndraws[b] = ndraws;
        if (out_flags) out_flags[b] = flags;
    }
    free(r);
    free(tst);
    free(dst);
}

/* ------------------------------------------------------------------------ */
/* orc_verify over the B sequences split into contiguous blocks, one per     */
/* thread (OpenMP when compiled with it; one after another otherwise).  Each */
/* block is orc_verify itself, keyed by the sequences' global indices (or    */
/* seq_ids), so the results equal one orc_verify call over all B: the        */
/* sequences of a step are independent.  Used to time the oracle on every    */
/* host core; the arithmetic is orc_verify's.                                */
/* ------------------------------------------------------------------------ */
void orc_verify_threads(int nthreads, int B, int K, int V, int dtype,
                        const void *target, const void *draft, const int32_t *draft_tokens,
                        const int32_t *draft_len, const int32_t *seq_ids, const float *temperature,
                        uint64_t seed, const double *theta,
                        int32_t *out_tokens, int32_t *out_accept_len,
                        double *out_feature, double *out_conf,
                        double *out_margin, int32_t *out_ndraws, int32_t *out_flags)
{
    size_t rowb = (size_t)V * (dtype == 0 ? 2 : 4);
    int nt = nthreads < 1 ? 1 : nthreads, t;
    if (nt > B) nt = B > 0 ? B : 1;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(static, 1)
#endif
    for (t = 0; t < nt; t++) {
        int b0 = (int)((long long)B * t / nt), b1 = (int)((long long)B * (t + 1) / nt), n = b1 - b0, i;
        int32_t *sid;
        if (n <= 0) continue;
        sid = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
        for (i = 0; i < n; i++) sid[i] = seq_ids ? seq_ids[b0 + i] : (int32_t)(b0 + i);
        orc_verify(n, K, V, dtype,
                   (const char *)target + (size_t)b0 * (size_t)(K + 1) * rowb,
                   (const char *)draft + (size_t)b0 * (size_t)K * rowb,
                   draft_tokens + (size_t)b0 * K, draft_len ? draft_len + b0 : NULL, sid, temperature + b0,
                   seed, theta, out_tokens + (size_t)b0 * (K + 1), out_accept_len + b0,
                   out_feature ? out_feature + (size_t)b0 * K : NULL, out_conf ? out_conf + (size_t)b0 * K : NULL,
                   out_margin ? out_margin + 2 * (size_t)b0 : NULL, out_ndraws ? out_ndraws + b0 : NULL,
                   out_flags ? out_flags + b0 : NULL);
        free(sid);
    }
}

/* ------------------------------------------------------------------------ */
/* [AV] "Fitting the coefficients".                                          */
/* Labels: drafts up to and including the first rejection; accepted = 1,     */
/* the rejected one = 0.  Accumulates the gradient g and Hessian H of the    */
/* summed log-loss at fixed theta, and the per-position label counts n.      */
/* H is dense (K+1)x(K+1), row-major; index 0 = omega, 1 + i = beta_i.       */
/* ------------------------------------------------------------------------ */
void orc_av_accumulate(int B, int K, const double *theta, const double *feature,
                       const int32_t *accept_len, const int32_t *kept_len,
                       double *g, double *H, double *n)
{
    int b, i, D = K + 1;
    for (b = 0; b < B; b++) {
        int a = accept_len[b];
        int k = kept_len ? kept_len[b] : K;
        int last;
        if (k > K) k = K;
        if (k < 0) k = 0;
        if (a > k) a = k;
        if (a < 0) a = 0;
        last = a < k ? a : a - 1; /* the rejected draft carries label 0 */
        for (i = 0; i <= last; i++) {
            double x = feature[(size_t)b * K + i];
            double y = i < a ? 1.0 : 0.0;
            double s = orc_conf(theta[0], theta[1 + i], x);
            double w = s * (1.0 - s);
            g[0] += (s - y) * x;
            g[1 + i] += (s - y);
            H[0 * D + 0] += w * x * x;
            H[0 * D + (1 + i)] += w * x;
            H[(1 + i) * D + 0] += w * x;
            H[(1 + i) * D + (1 + i)] += w;
            n[i] += 1.0;
        }
    }
}

/* Gaussian elimination with partial pivoting on the m x m system A z = rhs
 * (A and rhs are overwritten).  Returns 0 on success, 1 if singular. */
static int dense_solve(int m, double *A, double *rhs, double *z)
{
    int c, rr, cc;
    for (c = 0; c < m; c++) {
        int piv = c;
        double best = fabs(A[c * m + c]);
        for (rr = c + 1; rr < m; rr++)
            if (fabs(A[rr * m + c]) > best) { best = fabs(A[rr * m + c]); piv = rr; }
        if (best == 0.0) return 1;
        if (piv != c) {
            double t;
            for (cc = 0; cc < m; cc++) { t = A[c * m + cc]; A[c * m + cc] = A[piv * m + cc]; A[piv * m + cc] = t; }
            t = rhs[c]; rhs[c] = rhs[piv]; rhs[piv] = t;
        }
        for (rr = c + 1; rr < m; rr++) {
            double f = A[rr * m + c] / A[c * m + c];
            if (f == 0.0) continue;
            for (cc = c; cc < m; cc++) A[rr * m + cc] -= f * A[c * m + cc];
            rhs[rr] -= f * rhs[c];
        }
    }
    for (c = m - 1; c >= 0; c--) {
        double s = rhs[c];
        for (cc = c + 1; cc < m; cc++) s -= A[c * m + cc] * z[cc];
        z[c] = s / A[c * m + c];
    }
    return 0;
}

/* Newton (IRLS) step from accumulated (g, H, n): solve H delta = g over the
 * slope and the intercepts that have labels, with a ridge of
 * 1e-9 * trace(H) / (K+1) on the diagonal; then
 * theta_j <- theta_j - n_j / (n_j + c) * delta_j, n_omega = sum_i n_i.
 * Writes delta (K+1; 0 where dropped).  Returns 0 (updated), 1 (no labels),
 * 2 (singular). */
int orc_av_solve_update(int K, const double *g, const double *H, const double *n,
                        double damping_c, double *theta, double *delta)
{
    int D = K + 1, m = 0, i, j;
    int idx[64];
    double A[64 * 64], rhs[64], z[64];
    double trace = 0.0, ntot = 0.0, ridge;
    for (i = 0; i < D; i++) delta[i] = 0.0;
    for (i = 0; i < K; i++) ntot += n[i];
    if (ntot <= 0.0) return 1;
    idx[m++] = 0;
    for (i = 0; i < K; i++) if (n[i] > 0.0) idx[m++] = 1 + i;
    for (i = 0; i < D; i++) trace += H[i * D + i];
    ridge = 1e-9 * trace / (double)D;
    for (i = 0; i < m; i++) {
        for (j = 0; j < m; j++) A[i * m + j] = H[idx[i] * D + idx[j]];
        A[i * m + i] += ridge;
        rhs[i] = g[idx[i]];
    }
    if (dense_solve(m, A, rhs, z)) return 2;
    for (i = 0; i < m; i++) delta[idx[i]] = z[i];
    theta[0] -= ntot / (ntot + damping_c) * delta[0];
    for (i = 0; i < K; i++)
        if (n[i] > 0.0) theta[1 + i] -= n[i] / (n[i] + damping_c) * delta[1 + i];
    return 0;
}
