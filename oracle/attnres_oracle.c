/*
 * attnres_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * depth-wise softmax aggregation of Attention Residuals (AttnRes).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this library.  The CUDA
 * product path shares no code with it and never calls it.
 *
 * Every function follows the statement of the method on the pages, in their
 * order and notation:
 *   - "Attention Residual 深度残差" (K3 course notes, sec-09), eq. A1-A4,
 *     eq. OS1-OS2, listings "DepthResidual", "forward_naive",
 *     "_run_block_two_phase" and "atomic_block_size";
 *   - "Attention Residuals：当网络深度也拥有寻址能力", sections "Full AttnRes"
 *     and "Online softmax 让两阶段计算保持精确" (reference snippet
 *     depth_summary / merge_summary / finish).
 * Inputs are the exact values of the I/O tensors widened to double; the
 * query and gain are the fp32 parameters widened to double.  Rounding to
 * the I/O dtype happens only where the API hands a tensor back (a result
 * the caller can read), via oracle_round().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2   /* no rounding: the exact value is kept */

/* ---------------------------------------------------------------------- */
/* Rounding to the I/O dtype (round to nearest, ties to even).             */
/* ---------------------------------------------------------------------- */

/* bf16: 8 significant bits, fp32 exponent range (normal |x| >= 2^-126,
 * subnormal spacing 2^-133, largest finite (2 - 2^-7) * 2^127). */
double oracle_round_bf16(double x)
{
    if (!isfinite(x) || x == 0.0) return x;
    int e;
    (void)frexp(fabs(x), &e);            /* |x| = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                       /* exponent of one unit in the last place */
    if (q < -133) q = -133;              /* subnormal range */
    double r = rint(ldexp(x, -q));       /* rint: current mode, round-half-even */
    r = ldexp(r, q);
    if (fabs(r) >= ldexp(1.0, 128)) return x > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round_f32(double x) { return (double)(float)x; }

double oracle_round(double x, int dtype)
{
    if (dtype == ORACLE_F64) return x;
    return dtype == ORACLE_BF16 ? oracle_round_bf16(x) : oracle_round_f32(x);
}

void oracle_round_array(int64_t count, const double *x, int dtype, double *y)
{
    for (int64_t k = 0; k < count; ++k) y[k] = oracle_round(x[k], dtype);
}

/* ---------------------------------------------------------------------- */
/* Gain folding: w~ = w (.) gamma  ("DepthResidual", paragraph (1)).       */
/* gamma == NULL means a gain of one.                                     */
/* ---------------------------------------------------------------------- */
void oracle_fold_query(int64_t D, const double *w, const double *gamma, double *q_eff)
{
    for (int64_t d = 0; d < D; ++d) q_eff[d] = w[d] * (gamma ? gamma[d] : 1.0);
}

/* Gain-free RMS normalisation of one row: k = v / sqrt(mean_d v^2 + eps). */
static void rms_normalise(int64_t D, const double *v, double eps, double *k)
{
    double ss = 0.0;
    for (int64_t d = 0; d < D; ++d) ss += v[d] * v[d];
    double inv = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t d = 0; d < D; ++d) k[d] = v[d] * inv;
}

/* A1: s = w~^T RMS(v) for one row. */
static double depth_score(int64_t D, const double *q_eff, const double *v, double eps, double *kbuf)
{
    rms_normalise(D, v, eps, kbuf);
    double s = 0.0;
    for (int64_t d = 0; d < D; ++d) s += q_eff[d] * kbuf[d];
    return s;
}

/*
 * One token: A1 (scores on normalised sources), A2 (softmax over the source
 * axis), A3 (weighted sum of the RAW sources).  v[i] points at source i's
 * row of length D.  Outputs the unrounded h, the max score m and the
 * log-sum-exp lse = m + ln(sum_i exp(s_i - m)).
 */
static void aggregate_token(int n, int64_t D, const double *const *v, const double *q_eff,
                            double eps, double *h, double *m_out, double *lse_out,
                            double *scores, double *kbuf)
{
    for (int i = 0; i < n; ++i) scores[i] = depth_score(D, q_eff, v[i], eps, kbuf);
    double m = scores[0];
    for (int i = 1; i < n; ++i) if (scores[i] > m) m = scores[i];
    double z = 0.0;
    for (int i = 0; i < n; ++i) z += exp(scores[i] - m);
    for (int64_t d = 0; d < D; ++d) h[d] = 0.0;
    for (int i = 0; i < n; ++i) {
        double alpha = exp(scores[i] - m) / z;
        for (int64_t d = 0; d < D; ++d) h[d] += alpha * v[i][d];
    }
    if (m_out) *m_out = m;
    if (lse_out) *lse_out = m + log(z);
}

/*
 * Depth aggregation over n sources laid out as V[n][R][D] (R = B*T token
 * rows).  w, gamma: [D].  h: [R][D] unrounded; m, lse: [R] or NULL.
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_depth_aggregate(int n, int64_t R, int64_t D, const double *V, const double *w,
                           const double *gamma, double eps, double *h, double *m, double *lse)
{
    if (n < 1 || R < 0 || D < 1) return -1;
    double *q_eff = malloc(sizeof(double) * D);
    double *kbuf = malloc(sizeof(double) * D);
    double *scores = malloc(sizeof(double) * n);
    const double **rows = malloc(sizeof(double *) * n);
    if (!q_eff || !kbuf || !scores || !rows) { free(q_eff); free(kbuf); free(scores); free(rows); return -1; }
    oracle_fold_query(D, w, gamma, q_eff);
    for (int64_t r = 0; r < R; ++r) {
        for (int i = 0; i < n; ++i) rows[i] = V + ((int64_t)i * R + r) * D;
        aggregate_token(n, D, rows, q_eff, eps, h + r * D, m ? m + r : NULL, lse ? lse + r : NULL,
                        scores, kbuf);
    }
    free(q_eff); free(kbuf); free(scores); free(rows);
    return 0;
}

/*
 * Same as oracle_depth_aggregate, but the n sources are given as n separate
 * [R][D] arrays (the Full stack and the block recurrence keep a list of
 * sources, not a stacked tensor).
 */
int oracle_depth_aggregate_list(int n, int64_t R, int64_t D, const double *const *src,
                                const double *w, const double *gamma, double eps,
                                double *h, double *m, double *lse)
{
    if (n < 1 || R < 0 || D < 1) return -1;
    double *q_eff = malloc(sizeof(double) * D);
    double *kbuf = malloc(sizeof(double) * D);
    double *scores = malloc(sizeof(double) * n);
    const double **rows = malloc(sizeof(double *) * n);
    if (!q_eff || !kbuf || !scores || !rows) { free(q_eff); free(kbuf); free(scores); free(rows); return -1; }
    oracle_fold_query(D, w, gamma, q_eff);
    for (int64_t r = 0; r < R; ++r) {
        for (int i = 0; i < n; ++i) rows[i] = src[i] + r * D;
        aggregate_token(n, D, rows, q_eff, eps, h + r * D, m ? m + r : NULL, lse ? lse + r : NULL,
                        scores, kbuf);
    }
    free(q_eff); free(kbuf); free(scores); free(rows);
    return 0;
}

/*
 * Backward of the depth aggregation (the operator's backward pass that the
 * fused AttnRes operator computes by recomputation; "Attention Residuals：当
 * 网络深度也拥有寻址能力", sections "Depth attention 与 online merge reference"
 * and "公开实现边界").  The chain rule taken through the forward's steps in
 * reverse order, for each token row:
 *   A3  h = sum_i alpha_i v_i      ->  da_i = dh . v_i,   dv_i  = alpha_i dh
 *   A2  alpha = softmax(s)         ->  ds_i = alpha_i (da_i - sum_j alpha_j da_j)
 *   A1  s_i = q~ . k_i             ->  dq~ += ds_i k_i,   dk_i  = ds_i q~
 *   RMS k_i = v_i r_i, r_i = (mean_d v_i^2 + eps)^(-1/2)
 *                                  ->  dv_i += r_i dk_i - (r_i^3 / D)(v_i . dk_i) v_i
 * and, over all rows, the fold q~ = w (.) gamma  ->  dw = dq~ (.) gamma,
 * dgamma = dq~ (.) w.
 * src: n arrays [R][D]; dh: [R][D].  dV: n arrays [R][D] (overwritten).
 * dw: [D]; dgamma: [D] or NULL (only when gamma is given).
 */
int oracle_depth_aggregate_backward(int n, int64_t R, int64_t D, const double *const *src,
                                    const double *w, const double *gamma, double eps,
                                    const double *dh, double *const *dV, double *dw,
                                    double *dgamma)
{
    if (n < 1 || R < 0 || D < 1) return -1;
    double *q_eff = malloc(sizeof(double) * D);
    double *dq = calloc((size_t)D, sizeof(double));
    double *k = malloc(sizeof(double) * (size_t)n * D);
    double *r = malloc(sizeof(double) * n);
    double *s = malloc(sizeof(double) * n);
    double *alpha = malloc(sizeof(double) * n);
    double *da = malloc(sizeof(double) * n);
    if (!q_eff || !dq || !k || !r || !s || !alpha || !da) {
        free(q_eff); free(dq); free(k); free(r); free(s); free(alpha); free(da);
        return -1;
    }
    oracle_fold_query(D, w, gamma, q_eff);
    for (int64_t row = 0; row < R; ++row) {
        const double *g = dh + row * D;
        /* forward, recomputed: k_i, r_i, s_i, alpha_i */
        for (int i = 0; i < n; ++i) {
            const double *v = src[i] + row * D;
            double ss = 0.0;
            for (int64_t d = 0; d < D; ++d) ss += v[d] * v[d];
            r[i] = 1.0 / sqrt(ss / (double)D + eps);
            s[i] = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                k[(int64_t)i * D + d] = v[d] * r[i];
                s[i] += q_eff[d] * k[(int64_t)i * D + d];
            }
        }
        double m = s[0];
        for (int i = 1; i < n; ++i) if (s[i] > m) m = s[i];
        double z = 0.0;
        for (int i = 0; i < n; ++i) z += exp(s[i] - m);
        for (int i = 0; i < n; ++i) alpha[i] = exp(s[i] - m) / z;
        /* A3 */
        double mean_da = 0.0;
        for (int i = 0; i < n; ++i) {
            const double *v = src[i] + row * D;
            da[i] = 0.0;
            for (int64_t d = 0; d < D; ++d) da[i] += g[d] * v[d];
            mean_da += alpha[i] * da[i];
        }
        for (int i = 0; i < n; ++i) {
            const double *v = src[i] + row * D;
            double *dv = dV[i] + row * D;
            const double *ki = k + (int64_t)i * D;
            /* A2 */
            double ds = alpha[i] * (da[i] - mean_da);
            /* A1 */
            for (int64_t d = 0; d < D; ++d) dq[d] += ds * ki[d];
            /* RMS, with dk = ds q~ */
            double v_dot_dk = 0.0;
            for (int64_t d = 0; d < D; ++d) v_dot_dk += v[d] * ds * q_eff[d];
            double c = r[i] * r[i] * r[i] / (double)D * v_dot_dk;
            for (int64_t d = 0; d < D; ++d) dv[d] = alpha[i] * g[d] + r[i] * ds * q_eff[d] - c * v[d];
        }
    }
    for (int64_t d = 0; d < D; ++d) {
        dw[d] = dq[d] * (gamma ? gamma[d] : 1.0);
        if (dgamma) dgamma[d] = dq[d] * w[d];
    }
    free(q_eff); free(dq); free(k); free(r); free(s); free(alpha); free(da);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Online-softmax statistics (eq. OS1, OS2, single_source_stats).          */
/* A state is the triple (m, numer[D], denom) with h = numer / denom.      */
/* ---------------------------------------------------------------------- */

/* OS1 over a set of sources for one token. */
void oracle_os1_stats(int n, int64_t D, const double *const *v, const double *q_eff, double eps,
                      double *m_out, double *numer, double *denom_out)
{
    double *kbuf = malloc(sizeof(double) * D);
    double *s = malloc(sizeof(double) * n);
    for (int i = 0; i < n; ++i) s[i] = depth_score(D, q_eff, v[i], eps, kbuf);
    double m = s[0];
    for (int i = 1; i < n; ++i) if (s[i] > m) m = s[i];
    double den = 0.0;
    for (int64_t d = 0; d < D; ++d) numer[d] = 0.0;
    for (int i = 0; i < n; ++i) {
        double e = exp(s[i] - m);
        den += e;
        for (int64_t d = 0; d < D; ++d) numer[d] += e * v[i][d];
    }
    *m_out = m;
    *denom_out = den;
    free(kbuf); free(s);
}

/* single_source_stats: a lone source p has (m = s_p, numer = p, denom = 1). */
void oracle_single_source_stats(int64_t D, const double *p, const double *q_eff, double eps,
                                double *m_out, double *numer, double *denom_out)
{
    double *kbuf = malloc(sizeof(double) * D);
    *m_out = depth_score(D, q_eff, p, eps, kbuf);
    for (int64_t d = 0; d < D; ++d) numer[d] = p[d];
    *denom_out = 1.0;
    free(kbuf);
}

/* OS2: merge (m_a, n_a, d_a) and (m_b, n_b, d_b) into (m, n, d). */
void oracle_os2_merge(int64_t D, double m_a, const double *n_a, double d_a, double m_b,
                      const double *n_b, double d_b, double *m_out, double *n_out, double *d_out)
{
    double m = m_a > m_b ? m_a : m_b;
    double wa = exp(m_a - m), wb = exp(m_b - m);
    for (int64_t d = 0; d < D; ++d) n_out[d] = wa * n_a[d] + wb * n_b[d];
    *d_out = wa * d_a + wb * d_b;
    *m_out = m;
}

/* ---------------------------------------------------------------------- */
/* Two-phase Block inference ("两阶段算法（inter / intra）").              */
/* ---------------------------------------------------------------------- */

/*
 * Phase 1 (inter, batched): every one of the S queries of a block scores
 * the same n completed block summaries.  blocks: n arrays [R][D].
 * W, G: [S][D] (G may be NULL).  O: [S][R][D] unrounded, M, LSE: [S][R].
 */
int oracle_block_phase1(int n, int64_t R, int64_t D, const double *const *blocks, int S,
                        const double *W, const double *G, double eps, double *O, double *M,
                        double *LSE)
{
    for (int s = 0; s < S; ++s) {
        int rc = oracle_depth_aggregate_list(n, R, D, blocks, W + (int64_t)s * D,
                                             G ? G + (int64_t)s * D : NULL, eps,
                                             O + (int64_t)s * R * D, M ? M + (int64_t)s * R : NULL,
                                             LSE + (int64_t)s * R);
        if (rc) return rc;
    }
    return 0;
}

/*
 * Phase 2 (intra, one sublayer): merge the running partial p, as a single
 * source, into the phase-1 state of this sublayer's query, then normalise.
 * The phase-1 state is what phase 1 hands over: the normalised output o
 * and its log-sum-exp lse, i.e. the triple (lse, o, 1) -- the same state
 * as (m, numer, denom) rescaled so that denom = 1.
 * partial == NULL (first sublayer of a block): h = o.
 * h: [R][D] unrounded; lse_out: [R] merged log-sum-exp or NULL.
 */
int oracle_block_phase2_merge(int64_t R, int64_t D, const double *o, const double *lse,
                              const double *partial, const double *w, const double *gamma,
                              double eps, double *h, double *lse_out)
{
    double *q_eff = malloc(sizeof(double) * D);
    double *np = malloc(sizeof(double) * D);
    double *nm = malloc(sizeof(double) * D);
    if (!q_eff || !np || !nm) { free(q_eff); free(np); free(nm); return -1; }
    oracle_fold_query(D, w, gamma, q_eff);
    for (int64_t r = 0; r < R; ++r) {
        const double *orow = o + r * D;
        if (!partial) {
            for (int64_t d = 0; d < D; ++d) h[r * D + d] = orow[d];
            if (lse_out) lse_out[r] = lse[r];
            continue;
        }
        double mp, dp, mm, dm;
        oracle_single_source_stats(D, partial + r * D, q_eff, eps, &mp, np, &dp);
        oracle_os2_merge(D, lse[r], orow, 1.0, mp, np, dp, &mm, nm, &dm);
        for (int64_t d = 0; d < D; ++d) h[r * D + d] = nm[d] / dm;
        if (lse_out) lse_out[r] = mm + log(dm);
    }
    free(q_eff); free(np); free(nm);
    return 0;
}

/* Synthetic sublayer used by the benchmark recipes: f(h) = 0.5 * tanh(u (.) h). */
void oracle_synthetic_sublayer(int64_t R, int64_t D, const double *u, const double *h, double *out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t d = 0; d < D; ++d) out[r * D + d] = 0.5 * tanh(u[d] * h[r * D + d]);
}

/*
 * The next sublayer's pre-norm applied to h ("Attention Residuals：当网络深度
 * 也拥有寻址能力", sections "Depth attention 与 online merge reference" -- the
 * optional fused output RMSNorm -- and "Kimi Linear 与 K3 中的接入", where the
 * decode path fuses the merge, the partial update and the RMSNorm):
 *   y = x / sqrt(mean_d x^2 + eps) (.) weight      (weight == NULL: one)
 * row by row.  y may alias x.
 */
void oracle_rms_norm(int64_t R, int64_t D, const double *x, const double *weight, double eps,
                     double *y)
{
    for (int64_t r = 0; r < R; ++r) {
        double ss = 0.0;
        for (int64_t d = 0; d < D; ++d) ss += x[r * D + d] * x[r * D + d];
        double inv = 1.0 / sqrt(ss / (double)D + eps);
        for (int64_t d = 0; d < D; ++d) y[r * D + d] = x[r * D + d] * inv * (weight ? weight[d] : 1.0);
    }
}

/*
 * One block of the two-phase Block recurrence ("_run_block_two_phase")
 * with the synthetic sublayer:
 *   phase 1 over the n completed summaries for the block's S queries;
 *   for k = 1..S:  h_k = o_k (k = 1) or merge(o_k, lse_k, p_{k-1});
 *                  p_k = f_k(h_k) (k = 1) or p_{k-1} + f_k(h_k).
 * Rounding follows the tensors the API materialises: o_k (phase-1 output),
 * h_k (merge output, the sublayer's input) and p_k (the stored partial) are
 * rounded to the I/O dtype; lse stays fp32.
 * With NW ([S][D], the sublayers' pre-norm weights) the sublayer input is
 * y_k = rms_norm(h_k, NW_k, norm_eps), formed from the unrounded h_k; then
 * y_k is the materialised tensor (rounded) and h_k is not.
 * U: [S][D].  H_out: [S][R][D] rounded sublayer inputs (h_k, or y_k with NW);
 * P_out: [R][D] rounded p_S.
 */
int oracle_block_two_phase_chain(int n, int64_t R, int64_t D, const double *const *blocks, int S,
                                 const double *W, const double *G, const double *U,
                                 const double *NW, double norm_eps, double eps,
                                 int dtype, double *H_out, double *P_out)
{
    int64_t RD = R * D;
    double *O = malloc(sizeof(double) * (size_t)(S * RD));
    double *LSE = malloc(sizeof(double) * (size_t)(S * R));
    double *p = malloc(sizeof(double) * (size_t)RD);
    double *f = malloc(sizeof(double) * (size_t)RD);
    if (!O || !LSE || !p || !f) { free(O); free(LSE); free(p); free(f); return -1; }
    int rc = oracle_block_phase1(n, R, D, blocks, S, W, G, eps, O, NULL, LSE);
    if (rc) goto done;
    for (int64_t k = 0; k < S * RD; ++k) O[k] = oracle_round(O[k], dtype);
    /* lse is handed over as fp32 (exact in the F64 reference mode). */
    for (int64_t k = 0; k < S * R; ++k) LSE[k] = oracle_round(LSE[k], dtype == ORACLE_F64 ? ORACLE_F64 : ORACLE_F32);
    for (int s = 0; s < S; ++s) {
        double *hk = H_out + (int64_t)s * RD;
        rc = oracle_block_phase2_merge(R, D, O + (int64_t)s * RD, LSE + (int64_t)s * R,
                                       s == 0 ? NULL : p, W + (int64_t)s * D,
                                       G ? G + (int64_t)s * D : NULL, eps, hk, NULL);
        if (rc) goto done;
        if (NW) oracle_rms_norm(R, D, hk, NW + (int64_t)s * D, norm_eps, hk);
        for (int64_t k = 0; k < RD; ++k) hk[k] = oracle_round(hk[k], dtype);
        oracle_synthetic_sublayer(R, D, U + (int64_t)s * D, hk, f);
        for (int64_t k = 0; k < RD; ++k) p[k] = oracle_round((s == 0 ? 0.0 : p[k]) + f[k], dtype);
    }
    memcpy(P_out, p, sizeof(double) * (size_t)RD);
done:
    free(O); free(LSE); free(p); free(f);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* Block stack, naive form ("BlockAttnResStack.forward_naive"), in exact   */
/* fp64 with the synthetic sublayer; used to pin the two-phase form.       */
/* ---------------------------------------------------------------------- */

/*
 * N atomic sublayers, block size S (in sublayers).  x: [R][D] embedding.
 * W, G: [N+1][D] (row N is the final aggregate's query), U: [N][D].
 * NW: [N][D] pre-norm weights or NULL; with NW, sublayer idx reads
 * rms_norm(h, NW_idx, norm_eps) instead of h.
 * H_out: [N][R][D] (the input of every sublayer), y: [R][D] final.
 * Nothing is rounded: this is the exact reference the two-phase form must
 * reproduce.
 */
int oracle_block_forward_naive(int N, int S, int64_t R, int64_t D, const double *x,
                               const double *W, const double *G, const double *U,
                               const double *NW, double norm_eps, double eps,
                               double *H_out, double *y)
{
    int64_t RD = R * D;
    int max_blocks = N + 2;
    double **blocks = calloc((size_t)max_blocks, sizeof(double *));
    const double **srcs = calloc((size_t)max_blocks + 1, sizeof(double *));
    double *partial = malloc(sizeof(double) * (size_t)RD);
    double *out = malloc(sizeof(double) * (size_t)RD);
    int nb = 0, have_partial = 0, rc = 0;
    if (!blocks || !srcs || !partial || !out) { rc = -1; goto done; }
    blocks[nb] = malloc(sizeof(double) * (size_t)RD);
    memcpy(blocks[nb++], x, sizeof(double) * (size_t)RD);          /* b_0 = embedding */
    for (int idx = 1; idx <= N; ++idx) {
        int ns = 0;
        for (int b = 0; b < nb; ++b) srcs[ns++] = blocks[b];
        if (have_partial) srcs[ns++] = partial;
        double *h = H_out + (int64_t)(idx - 1) * RD;
        rc = oracle_depth_aggregate_list(ns, R, D, srcs, W + (int64_t)(idx - 1) * D,
                                         G ? G + (int64_t)(idx - 1) * D : NULL, eps, h, NULL, NULL);
        if (rc) goto done;
        if (NW) oracle_rms_norm(R, D, h, NW + (int64_t)(idx - 1) * D, norm_eps, h);
        oracle_synthetic_sublayer(R, D, U + (int64_t)(idx - 1) * D, h, out);
        for (int64_t k = 0; k < RD; ++k) partial[k] = have_partial ? partial[k] + out[k] : out[k];
        have_partial = 1;
        if (idx % S == 0 || idx == N) {                               /* block boundary */
            blocks[nb] = malloc(sizeof(double) * (size_t)RD);
            memcpy(blocks[nb++], partial, sizeof(double) * (size_t)RD);
            have_partial = 0;
        }
    }
    for (int b = 0; b < nb; ++b) srcs[b] = blocks[b];
    rc = oracle_depth_aggregate_list(nb, R, D, srcs, W + (int64_t)N * D,
                                     G ? G + (int64_t)N * D : NULL, eps, y, NULL, NULL);
done:
    if (blocks) for (int b = 0; b < nb; ++b) free(blocks[b]);
    free(blocks); free(srcs); free(partial); free(out);
    return rc;
}

/*
 * Block stack, two-phase form ("_run_block_two_phase"), exact fp64, same
 * arguments as the naive form.  Each block runs phase 1 once over the
 * completed summaries, then merges the running partial sublayer by
 * sublayer.  The phase-1 state is carried as the full triple (m, numer,
 * denom), nothing rounded.
 */
int oracle_block_forward_two_phase(int N, int S, int64_t R, int64_t D, const double *x,
                                   const double *W, const double *G, const double *U, double eps,
                                   double *H_out, double *y)
{
    int64_t RD = R * D;
    int max_blocks = N + 2;
    double **blocks = calloc((size_t)max_blocks, sizeof(double *));
    double *partial = malloc(sizeof(double) * (size_t)RD);
    double *out = malloc(sizeof(double) * (size_t)RD);
    double *q_eff = malloc(sizeof(double) * (size_t)D);
    double *n1 = malloc(sizeof(double) * (size_t)D);
    double *np = malloc(sizeof(double) * (size_t)D);
    double *nm = malloc(sizeof(double) * (size_t)D);
    const double **rows = calloc((size_t)max_blocks, sizeof(double *));
    int nb = 0, rc = 0;
    if (!blocks || !partial || !out || !q_eff || !n1 || !np || !nm || !rows) { rc = -1; goto done; }
    blocks[nb] = malloc(sizeof(double) * (size_t)RD);
    memcpy(blocks[nb++], x, sizeof(double) * (size_t)RD);
    for (int start = 0; start < N; start += S) {
        int end = start + S < N ? start + S : N;
        for (int li = start; li < end; ++li) {
            oracle_fold_query(D, W + (int64_t)li * D, G ? G + (int64_t)li * D : NULL, q_eff);
            double *h = H_out + (int64_t)li * RD;
            for (int64_t r = 0; r < R; ++r) {
                double m1, d1;
                for (int b = 0; b < nb; ++b) rows[b] = blocks[b] + r * D;
                oracle_os1_stats(nb, D, rows, q_eff, eps, &m1, n1, &d1);   /* phase 1 */
                if (li > start) {                                          /* phase 2 */
                    double mp, dp, mm, dm;
                    oracle_single_source_stats(D, partial + r * D, q_eff, eps, &mp, np, &dp);
                    oracle_os2_merge(D, m1, n1, d1, mp, np, dp, &mm, nm, &dm);
                    for (int64_t d = 0; d < D; ++d) h[r * D + d] = nm[d] / dm;
                } else {
                    for (int64_t d = 0; d < D; ++d) h[r * D + d] = n1[d] / d1;
                }
            }
            oracle_synthetic_sublayer(R, D, U + (int64_t)li * D, h, out);
            for (int64_t k = 0; k < RD; ++k) partial[k] = li > start ? partial[k] + out[k] : out[k];
        }
        blocks[nb] = malloc(sizeof(double) * (size_t)RD);
        memcpy(blocks[nb++], partial, sizeof(double) * (size_t)RD);
    }
    {
        const double **srcs = (const double **)blocks;
        rc = oracle_depth_aggregate_list(nb, R, D, srcs, W + (int64_t)N * D,
                                         G ? G + (int64_t)N * D : NULL, eps, y, NULL, NULL);
    }
done:
    if (blocks) for (int b = 0; b < nb; ++b) free(blocks[b]);
    free(blocks); free(partial); free(out); free(q_eff); free(n1); free(np); free(nm); free(rows);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* Full stack ("FullAttnResStack", eq. A1-A4) with the synthetic sublayer.  */
/* ---------------------------------------------------------------------- */

/*
 * L sublayers.  v0: [R][D] (given, exact).  W, G: [L+1][D] (row L is the
 * final aggregate's query), U: [L][D].  V_out: [L+1][R][D]; row 0 is v0,
 * rows 1..L are v_l = round(0.5 tanh(u_l (.) h_l)) with h_l the unrounded
 * aggregate over v_0..v_{l-1}.  y: [R][D] unrounded final aggregate over
 * v_0..v_L.
 */
int oracle_full_stack_forward(int L, int64_t R, int64_t D, const double *v0, const double *W,
                              const double *G, const double *U, double eps, int dtype,
                              double *V_out, double *y)
{
    int64_t RD = R * D;
    const double **srcs = malloc(sizeof(double *) * (size_t)(L + 1));
    double *h = malloc(sizeof(double) * (size_t)RD);
    int rc = 0;
    if (!srcs || !h) { free(srcs); free(h); return -1; }
    memcpy(V_out, v0, sizeof(double) * (size_t)RD);
    for (int l = 0; l <= L; ++l) srcs[l] = V_out + (int64_t)l * RD;
    for (int l = 1; l <= L; ++l) {
        rc = oracle_depth_aggregate_list(l, R, D, srcs, W + (int64_t)(l - 1) * D,
                                         G ? G + (int64_t)(l - 1) * D : NULL, eps, h, NULL, NULL);
        if (rc) break;
        double *vl = V_out + (int64_t)l * RD;
        oracle_synthetic_sublayer(R, D, U + (int64_t)(l - 1) * D, h, vl);
        for (int64_t k = 0; k < RD; ++k) vl[k] = oracle_round(vl[k], dtype);
    }
    if (!rc)
        rc = oracle_depth_aggregate_list(L + 1, R, D, srcs, W + (int64_t)L * D,
                                         G ? G + (int64_t)L * D : NULL, eps, y, NULL, NULL);
    free(srcs); free(h);
    return rc;
}

/*
 * Full stack with the two-phase schedule (a schedule block size S: the
 * remark under "_run_block_two_phase" that Full AttnRes runs two-phase when
 * schedule_block_size is given, and the (S+N)d residual I/O of "推理：block
 * representations 像一份 depth KV cache").  Sublayers are taken S at a time;
 * for the block of sublayers l = start+1 .. min(start+S, L):
 *   phase 1: for every l of the block, the OS1 state of query l over the
 *            sources completed before the block, v_0 .. v_start, handed over
 *            normalised as (lse_l, o_l, 1);
 *   phase 2: in order, h_l = that state merged (OS2) with each intra-block
 *            source v_{start+1} .. v_{l-1} (single_source_stats), and
 *            v_l = f_l(h_l) with the synthetic sublayer.
 * The final aggregate is the plain one over v_0 .. v_L.  Rounding follows
 * what the GPU path materialises: o_l to the I/O dtype (lse as fp32) and
 * v_l to the I/O dtype; h_l stays unrounded (f is fused).  In the F64 mode
 * nothing is rounded and the result equals oracle_full_stack_forward's.
 * Arguments as oracle_full_stack_forward, plus S >= 1.
 */
int oracle_full_stack_two_phase(int L, int S, int64_t R, int64_t D, const double *v0, const double *W,
                                const double *G, const double *U, double eps, int dtype,
                                double *V_out, double *y)
{
    if (L < 1 || S < 1 || R < 0 || D < 1) return -1;
    int64_t RD = R * D;
    const double **srcs = malloc(sizeof(double *) * (size_t)(L + 1));
    const double **rows = malloc(sizeof(double *) * (size_t)(L + 1));
    double *O = malloc(sizeof(double) * (size_t)S * (size_t)RD);
    double *LSE = malloc(sizeof(double) * (size_t)S * (size_t)R);
    double *q_eff = malloc(sizeof(double) * (size_t)D);
    double *numer = malloc(sizeof(double) * (size_t)D);
    double *np = malloc(sizeof(double) * (size_t)D);
    double *nm = malloc(sizeof(double) * (size_t)D);
    double *h = malloc(sizeof(double) * (size_t)RD);
    int rc = 0;
    if (!srcs || !rows || !O || !LSE || !q_eff || !numer || !np || !nm || !h) { rc = -1; goto done; }
    memcpy(V_out, v0, sizeof(double) * (size_t)RD);
    for (int l = 0; l <= L; ++l) srcs[l] = V_out + (int64_t)l * RD;
    for (int start = 0; start < L; start += S) {
        int end = start + S < L ? start + S : L;          /* sublayers start+1 .. end */
        /* phase 1: every query of the block over v_0 .. v_start */
        for (int l = start + 1; l <= end; ++l) {
            int s = l - start - 1;
            oracle_fold_query(D, W + (int64_t)(l - 1) * D, G ? G + (int64_t)(l - 1) * D : NULL, q_eff);
            for (int64_t r = 0; r < R; ++r) {
                double m1, d1;
                for (int i = 0; i <= start; ++i) rows[i] = srcs[i] + r * D;
                oracle_os1_stats(start + 1, D, rows, q_eff, eps, &m1, numer, &d1);
                double *o = O + ((int64_t)s * R + r) * D;
                for (int64_t d = 0; d < D; ++d) o[d] = oracle_round(numer[d] / d1, dtype);
                LSE[(int64_t)s * R + r] = oracle_round(m1 + log(d1), dtype == ORACLE_F64 ? ORACLE_F64 : ORACLE_F32);
            }
        }
        /* phase 2: in order, merge the intra-block sources, then the sublayer */
        for (int l = start + 1; l <= end; ++l) {
            int s = l - start - 1;
            oracle_fold_query(D, W + (int64_t)(l - 1) * D, G ? G + (int64_t)(l - 1) * D : NULL, q_eff);
            for (int64_t r = 0; r < R; ++r) {
                double m = LSE[(int64_t)s * R + r], den = 1.0;
                for (int64_t d = 0; d < D; ++d) numer[d] = O[((int64_t)s * R + r) * D + d];
                for (int j = start + 1; j < l; ++j) {
                    double mp, dp, mm, dm;
                    oracle_single_source_stats(D, srcs[j] + r * D, q_eff, eps, &mp, np, &dp);
                    oracle_os2_merge(D, m, numer, den, mp, np, dp, &mm, nm, &dm);
                    m = mm;
                    den = dm;
                    memcpy(numer, nm, sizeof(double) * (size_t)D);
                }
                for (int64_t d = 0; d < D; ++d) h[r * D + d] = numer[d] / den;
            }
            double *vl = V_out + (int64_t)l * RD;
            oracle_synthetic_sublayer(R, D, U + (int64_t)(l - 1) * D, h, vl);
            for (int64_t k = 0; k < RD; ++k) vl[k] = oracle_round(vl[k], dtype);
        }
    }
    rc = oracle_depth_aggregate_list(L + 1, R, D, srcs, W + (int64_t)L * D,
                                     G ? G + (int64_t)L * D : NULL, eps, y, NULL, NULL);
done:
    free(srcs); free(rows); free(O); free(LSE); free(q_eff); free(numer); free(np); free(nm); free(h);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* Bookkeeping ("forward_naive" source lists, "atomic_block_size").        */
/* ---------------------------------------------------------------------- */

/*
 * DecoderBlocks -> atomic sublayers per AttnRes block.  has_block_size = 0
 * is the "None" of the config field: about eight blocks, ceil(L/8)
 * DecoderBlocks each, at least one.  Each DecoderBlock is two atomic
 * sublayers (attention and FFN).
 */
int oracle_atomic_block_size(int num_hidden_layers, int has_block_size, int block_size)
{
    int layers_per_block;
    if (has_block_size) {
        layers_per_block = block_size;
    } else {
        layers_per_block = (num_hidden_layers + 7) / 8;
        if (layers_per_block < 1) layers_per_block = 1;
    }
    return layers_per_block * 2;
}

/*
 * Replays forward_naive's list handling for N atomic sublayers and block
 * size S.  Writes, for every sublayer and then for the final aggregate,
 * the ids of the sources it sees: block ids 0.. (0 = embedding) and -1
 * for the running partial.  counts: [N+1].  ids: flat, capacity entries.
 * Returns the number of ids written, or -1 if capacity is too small.
 */
int oracle_block_schedule(int N, int S, int *counts, int *ids, int capacity)
{
    int nb = 1, have_partial = 0, w = 0;          /* blocks = [x] */
    for (int idx = 1; idx <= N; ++idx) {
        int c = 0;
        for (int b = 0; b < nb; ++b) { if (w >= capacity) return -1; ids[w++] = b; ++c; }
        if (have_partial) { if (w >= capacity) return -1; ids[w++] = -1; ++c; }
        counts[idx - 1] = c;
        have_partial = 1;                          /* partial = out or partial + out */
        if (idx % S == 0 || idx == N) { ++nb; have_partial = 0; }
    }
    for (int b = 0; b < nb; ++b) { if (w >= capacity) return -1; ids[w++] = b; }
    counts[N] = nb;
    return w;
}
