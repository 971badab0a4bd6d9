/*
 * attn_ref.c -- FP64 CPU oracle for dense scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header or constant with the CUDA path.
 *
 * What it computes is the plain definition written out, one query row at a time,
 * with no tiling and no online recurrence:
 *
 *   S = scale * Q K^T,   P = softmax_row(S),   O = P V
 *
 * ("FlashAttention'ı Anlamak Bölüm 1", section 0.2 Notasyon, with the optional
 * mask/bias B taken as zero here, as the causal mask and as a caller-given bias in
 * the two functions that say so; the scale is the caller's, applied to the scores as
 * in the "Алгоритм Flash Attention 2" pseudocode of "Flash Attention на 5090 в
 * CUDA C++"). The same notes (section 0.1) state that FlashAttention reaches this
 * exact result, only in a different floating-point order, so a tiled GPU kernel
 * must agree with it up to rounding.
 *
 * Per query row i of head (b,h), in double precision from BF16 inputs widened
 * exactly:
 *   1. s_j = scale * sum_c q[i,c] * k[j,c]           for every key j
 *   2. m   = max_j s_j
 *   3. l   = sum_j exp(s_j - m)
 *   4. o_c = (sum_j exp(s_j - m) * v[j,c]) / l
 *   5. lse = m + log(l)     (natural log of sum_j exp(s_j))
 * Subtracting m leaves P unchanged (the common factor exp(-m) cancels) and keeps
 * exp() from overflowing; step 5 adds it back.
 *
 * The log-sum-exp output is not defined on the pages; it is read here as the
 * natural logarithm of the softmax denominator in scaled-score units, one value
 * per query row.
 *
 * Parity pins for every function below live in tests/test_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes of this file (independent of the library's own). */
#define REF_OK 0
#define REF_EINVAL (-1)
#define REF_ENOMEM (-2)

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* step 1: s_j = scale * (q_i . k_j) for every key j of one head */
static void row_scores(const uint16_t *qi, const uint16_t *kh, int64_t Nk, int64_t d,
                       double scale, double *s)
{
    for (int64_t j = 0; j < Nk; j++) {
        const uint16_t *kj = kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; c++)
            acc += bf16_to_f64(qi[c]) * bf16_to_f64(kj[c]);
        s[j] = scale * acc;
    }
}

/* step 2: m = max_j s_j */
static double row_max(const double *s, int64_t Nk)
{
    double m = s[0];
    for (int64_t j = 1; j < Nk; j++)
        if (s[j] > m) m = s[j];
    return m;
}

/* step 3: overwrite s_j with exp(s_j - m) and return their sum l */
static double row_exp_sum(double *s, int64_t Nk, double m)
{
    double l = 0.0;
    for (int64_t j = 0; j < Nk; j++) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    return l;
}

/*
 * One query row i: writes o[0..dv) and *lse. s is caller scratch of Nk doubles.
 * bh_bias, when not NULL, is the head's additive bias B: B_ij = bh_bias[i * sq + j].
 */
static void attend_row(const uint16_t *qi, const uint16_t *kh, const uint16_t *vh,
                       const uint16_t *bh_bias, int64_t i, int64_t sq,
                       int64_t Nk, int64_t d, int64_t dv, double scale,
                       double *s, double *o, double *lse)
{
    row_scores(qi, kh, Nk, d, scale, s);
    if (bh_bias) {   /* S = scale * Q K^T + B */
        for (int64_t j = 0; j < Nk; j++)
            s[j] += bf16_to_f64(bh_bias[i * sq + j]);
    }
    double m = row_max(s, Nk);
    double l = row_exp_sum(s, Nk, m);
    /* step 4: weighted sum of value rows */
    for (int64_t c = 0; c < dv; c++) {
        double acc = 0.0;
        for (int64_t j = 0; j < Nk; j++)
            acc += s[j] * bf16_to_f64(vh[j * dv + c]);
        o[c] = acc / l;
    }
    /* step 5 */
    *lse = m + log(l);
}

/*
 * attn_ref_rows_f64: O and LSE for a chosen set of query rows.
 *
 *   q   [BH, Nq, d]   BF16 bit patterns, C order     (BH = batch * heads)
 *   k   [BH, Nk, d]
 *   v   [BH, Nk, dv]
 *   sel [nsel]        flat row ids bh*Nq + i, each in [0, BH*Nq)
 *   o   [nsel, dv]    output, float64
 *   lse [nsel]        output, float64
 *   nthreads          OpenMP threads (<= 0: the runtime's default)
 *
 * Returns REF_OK, REF_EINVAL for a bad size or row id, REF_ENOMEM.
 */
int attn_ref_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                      double scale, const int64_t *sel, int64_t nsel,
                      double *o, double *lse, int nthreads)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || nsel < 0) return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q || !k || !v || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                attend_row(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * dv,
                           NULL, i, 0, Nk, d, dv, scale, s, o + r * dv, lse + r);
            }
            free(s);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

/*
 * attn_ref_rows_causal_f64: O and LSE of selected rows under the causal mask.
 *
 * The definition's optional mask B ("FlashAttention'ı Anlamak Bölüm 1", section 0.2)
 * taken as the causal mask, aligned to the bottom-right corner of the score matrix:
 * B_ij = 0 when j <= i + (Nk - Nq) and -inf otherwise, so that the last query row sees
 * every key (the layout of a query block appended after Nk - Nq earlier positions).
 * exp(-inf) = 0 removes a masked key from both sums, so row i is exactly the plain
 * definition over its visible keys 0 .. i + Nk - Nq, which is how it is computed here.
 * Requires Nq <= Nk (every row sees at least one key). Arguments as attn_ref_rows_f64.
 */
int attn_ref_rows_causal_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                             double scale, const int64_t *sel, int64_t nsel,
                             double *o, double *lse, int nthreads)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || nsel < 0 || Nq > Nk) return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q || !k || !v || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                int64_t visible = i + (Nk - Nq) + 1;   /* keys 0 .. i + Nk - Nq */
                attend_row(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * dv,
                           NULL, i, 0, visible, d, dv, scale, s, o + r * dv, lse + r);
            }
            free(s);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

/*
 * attn_ref_rows_bias_f64: O and LSE of selected rows with an additive bias.
 *
 * The definition's S = Q K^T / sqrt(d) + B, P = softmax_row(S), O = P V
 * ("FlashAttention'ı Anlamak Bölüm 1", section 0.2 Notasyon), with the caller's scale
 * in place of 1/sqrt(d) as above and B given per head as BF16 bit patterns:
 *
 *   B_ij of head (b, h) = bias[b * sb + h * sh + i * sq + j]     (strides in elements)
 *
 * A stride of 0 repeats the same values across batches, heads or query rows (sq = 0:
 * one bias per key, e.g. a padding mask). An entry of -inf removes that key from the
 * row (exp(-inf) = 0); a row whose entries are all -inf has no softmax, and its O and
 * LSE come out NaN. H is the number of heads per batch (BH = B * H). Other arguments as
 * attn_ref_rows_f64.
 */
int attn_ref_rows_bias_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const uint16_t *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq,
                           int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                           double scale, const int64_t *sel, int64_t nsel,
                           double *o, double *lse, int nthreads)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || nsel < 0) return REF_EINVAL;
    if (H < 1 || BH % H != 0 || sb < 0 || sh < 0 || sq < 0) return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q || !k || !v || !bias || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                const uint16_t *bh_bias = bias + (bh / H) * sb + (bh % H) * sh;
                attend_row(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * dv,
                           bh_bias, i, sq, Nk, d, dv, scale, s, o + r * dv, lse + r);
            }
            free(s);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

/*
 * attn_ref_probs_f64: the full probability matrix P = softmax_row(scale * Q K^T),
 * p [BH, Nq, Nk], for small shapes (tests of the row normalisation).
 */
int attn_ref_probs_f64(const uint16_t *q, const uint16_t *k,
                       int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                       double scale, double *p)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1) return REF_EINVAL;
    if (BH * Nq == 0) return REF_OK;
    if (!q || !k || !p) return REF_EINVAL;
    for (int64_t bh = 0; bh < BH; bh++) {
        for (int64_t i = 0; i < Nq; i++) {
            double *s = p + (bh * Nq + i) * Nk;
            row_scores(q + (bh * Nq + i) * d, k + bh * Nk * d, Nk, d, scale, s);
            double m = row_max(s, Nk);
            double l = row_exp_sum(s, Nk, m);
            for (int64_t j = 0; j < Nk; j++) s[j] /= l;
        }
    }
    return REF_OK;
}

/* Number of threads an OpenMP region of this library would use by default. */
int attn_ref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * ---- Backward pass ---------------------------------------------------------------
 *
 * The notes name the backward pass and recomputation as parts of the method
 * ("FlashAttention'ı Anlamak Bölüm 1", section 0 Giriş: tiling, online softmax and
 * recomputation; forward and backward passes) without giving its formulas. What it
 * computes is fixed by the mathematics: the gradient of the forward above for a loss L
 * whose gradient with respect to O is dO. Row by row, in double precision:
 *
 *   p_j   = exp(s_j - m) / l                     (the forward's probabilities, recomputed)
 *   dv_j += p_j * dO_i                           (O_i = sum_j p_j v_j)
 *   dp_j  = dO_i . v_j
 *   D_i   = sum_j p_j dp_j                       (= dO_i . O_i)
 *   ds_j  = p_j (dp_j - D_i)                     (softmax Jacobian: dp/ds = diag(p) - p p^T)
 *   dq_i  = scale * sum_j ds_j k_j               (s_j = scale * q_i . k_j)
 *   dk_j += scale * ds_j q_i
 *
 * These take double inputs so that central differences of attn_ref_dense_f64 can check
 * them; BF16 inputs are widened exactly by the caller.
 *
 * With the definition's optional bias B (section 0.2: S = QK^T / sqrt(d) + B), held fixed,
 * s_j = scale * q_i . k_j + B_ij and every formula above is unchanged: B enters the
 * gradients only through p (a constant's derivative is zero), and dB = ds is not formed.
 * The bias arrives as doubles, B_ij of head (b, h) = bias[b * sb + h * sh + i * sq + j].
 */
struct dbias { const double *p; int64_t H, sb, sh, sq; };   /* p == NULL: no bias */

/* row i of head bh's bias, or NULL */
static const double *dbias_row(const struct dbias *b, int64_t bh, int64_t i)
{
    return b->p ? b->p + (bh / b->H) * b->sb + (bh % b->H) * b->sh + i * b->sq : NULL;
}

static int dbias_ok(const struct dbias *b, int64_t BH)
{
    return !b->p || (b->H >= 1 && BH % b->H == 0 && b->sb >= 0 && b->sh >= 0 && b->sq >= 0);
}

/*
 * The forward on double inputs: o [BH, Nq, dv], lse [BH, Nq] (same steps as above).
 * causal != 0: row i uses keys 0 .. i + (Nk - Nq) only (the causal mask of
 * attn_ref_rows_causal_f64; needs Nq <= Nk).
 */
static int dense_impl(const double *q, const double *k, const double *v,
                      int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                      double scale, double *o, double *lse, int causal, const struct dbias *bias)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1) return REF_EINVAL;
    if ((causal && Nq > Nk) || !dbias_ok(bias, BH)) return REF_EINVAL;
    if (BH * Nq == 0) return REF_OK;
    if (!q || !k || !v || !o || !lse) return REF_EINVAL;
    double *s = (double *)malloc((size_t)Nk * sizeof(double));
    if (!s) return REF_ENOMEM;
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *kh = k + bh * Nk * d, *vh = v + bh * Nk * dv;
        for (int64_t i = 0; i < Nq; i++) {
            const double *qi = q + (bh * Nq + i) * d;
            const int64_t nv = causal ? i + (Nk - Nq) + 1 : Nk;   /* keys of row i */
            for (int64_t j = 0; j < nv; j++) {
                double acc = 0.0;
                for (int64_t c = 0; c < d; c++) acc += qi[c] * kh[j * d + c];
                s[j] = scale * acc;
            }
            const double *bi = dbias_row(bias, bh, i);
            if (bi)
                for (int64_t j = 0; j < nv; j++) s[j] += bi[j];
            double m = row_max(s, nv);
            double l = row_exp_sum(s, nv, m);
            double *oi = o + (bh * Nq + i) * dv;
            for (int64_t c = 0; c < dv; c++) {
                double acc = 0.0;
                for (int64_t j = 0; j < nv; j++) acc += s[j] * vh[j * dv + c];
                oi[c] = acc / l;
            }
            lse[bh * Nq + i] = m + log(l);
        }
    }
    free(s);
    return REF_OK;
}

int attn_ref_dense_f64(const double *q, const double *k, const double *v,
                       int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                       double scale, double *o, double *lse)
{
    const struct dbias none = {NULL, 1, 0, 0, 0};
    return dense_impl(q, k, v, BH, Nq, Nk, d, dv, scale, o, lse, 0, &none);
}

int attn_ref_dense_causal_f64(const double *q, const double *k, const double *v,
                              int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                              double scale, double *o, double *lse)
{
    const struct dbias none = {NULL, 1, 0, 0, 0};
    return dense_impl(q, k, v, BH, Nq, Nk, d, dv, scale, o, lse, 1, &none);
}

/* the forward on double inputs with the bias (no causal mask: a bias can carry one) */
int attn_ref_dense_bias_f64(const double *q, const double *k, const double *v,
                            const double *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq,
                            int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                            double scale, double *o, double *lse)
{
    if (!bias) return REF_EINVAL;
    const struct dbias b = {bias, H, sb, sh, sq};
    return dense_impl(q, k, v, BH, Nq, Nk, d, dv, scale, o, lse, 0, &b);
}

/*
 * attn_ref_bwd_f64: dq [BH, Nq, d], dk [BH, Nk, d], dv [BH, Nk, dv] for upstream
 * gradient dout [BH, Nq, dv]. OpenMP over heads (each head's dk and dv are summed over
 * its query rows in order). causal != 0 (attn_ref_bwd_causal_f64): the gradient of the
 * causal forward, every sum of row i running over its keys 0 .. i + (Nk - Nq) only.
 */
static int bwd_impl(const double *q, const double *k, const double *v, const double *dout,
                    int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                    double scale, double *dq, double *dk, double *dvv, int nthreads, int causal,
                    const struct dbias *bias)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1) return REF_EINVAL;
    if ((causal && Nq > Nk) || !dbias_ok(bias, BH)) return REF_EINVAL;
    if (BH == 0) return REF_OK;
    if (!q || !k || !v || !dout || !dq || !dk || !dvv) return REF_EINVAL;
    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *p = (double *)malloc((size_t)Nk * sizeof(double));
        double *dp = (double *)malloc((size_t)Nk * sizeof(double));
        if (!p || !dp) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t bh = 0; bh < BH; bh++) {
                const double *kh = k + bh * Nk * d, *vh = v + bh * Nk * dv;
                double *dkh = dk + bh * Nk * d, *dvh = dvv + bh * Nk * dv;
                memset(dkh, 0, (size_t)(Nk * d) * sizeof(double));
                memset(dvh, 0, (size_t)(Nk * dv) * sizeof(double));
                for (int64_t i = 0; i < Nq; i++) {
                    const double *qi = q + (bh * Nq + i) * d;
                    const double *doi = dout + (bh * Nq + i) * dv;
                    double *dqi = dq + (bh * Nq + i) * d;
                    const int64_t nvis = causal ? i + (Nk - Nq) + 1 : Nk;   /* keys of row i */
                    /* the forward's probabilities of row i */
                    for (int64_t j = 0; j < nvis; j++) {
                        double acc = 0.0;
                        for (int64_t c = 0; c < d; c++) acc += qi[c] * kh[j * d + c];
                        p[j] = scale * acc;
                    }
                    const double *brow = dbias_row(bias, bh, i);
                    if (brow)
                        for (int64_t j = 0; j < nvis; j++) p[j] += brow[j];
                    double m = row_max(p, nvis);
                    double l = row_exp_sum(p, nvis, m);
                    for (int64_t j = 0; j < nvis; j++) p[j] /= l;
                    /* dv, dp and D */
                    double D = 0.0;
                    for (int64_t j = 0; j < nvis; j++) {
                        double acc = 0.0;
                        for (int64_t c = 0; c < dv; c++) {
                            dvh[j * dv + c] += p[j] * doi[c];
                            acc += doi[c] * vh[j * dv + c];
                        }
                        dp[j] = acc;
                        D += p[j] * acc;
                    }
                    /* ds, dq, dk */
                    for (int64_t c = 0; c < d; c++) dqi[c] = 0.0;
                    for (int64_t j = 0; j < nvis; j++) {
                        double ds = p[j] * (dp[j] - D);
                        for (int64_t c = 0; c < d; c++) {
                            dqi[c] += scale * ds * kh[j * d + c];
                            dkh[j * d + c] += scale * ds * qi[c];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? REF_ENOMEM : REF_OK;
}

int attn_ref_bwd_f64(const double *q, const double *k, const double *v, const double *dout,
                     int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                     double scale, double *dq, double *dk, double *dvv, int nthreads)
{
    const struct dbias none = {NULL, 1, 0, 0, 0};
    return bwd_impl(q, k, v, dout, BH, Nq, Nk, d, dv, scale, dq, dk, dvv, nthreads, 0, &none);
}

int attn_ref_bwd_causal_f64(const double *q, const double *k, const double *v, const double *dout,
                            int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                            double scale, double *dq, double *dk, double *dvv, int nthreads)
{
    const struct dbias none = {NULL, 1, 0, 0, 0};
    return bwd_impl(q, k, v, dout, BH, Nq, Nk, d, dv, scale, dq, dk, dvv, nthreads, 1, &none);
}

/* the gradient (dq, dk, dv) of the biased forward, the bias held fixed */
int attn_ref_bwd_bias_f64(const double *q, const double *k, const double *v, const double *dout,
                          const double *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq,
                          int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                          double scale, double *dq, double *dk, double *dvv, int nthreads)
{
    if (!bias) return REF_EINVAL;
    const struct dbias b = {bias, H, sb, sh, sq};
    return bwd_impl(q, k, v, dout, BH, Nq, Nk, d, dv, scale, dq, dk, dvv, nthreads, 0, &b);
}

/*
 * FP8 E4M3 scores.
 *
 * "Flash Attention на 5090 в CUDA C++" (section "Что дальше") names low-precision (FP8)
 * MMA as the next step. Read plainly: Q and K arrive as 8-bit E4M3 codes with one
 * descale factor per tensor, the real inputs being q_descale * Q8 and k_descale * K8,
 * and the definition above is applied to them unchanged:
 *   s_j = scale * sum_c (q_descale * q8[i,c]) * (k_descale * k8[j,c]),
 * then steps 2-5 with V in BF16.
 *
 * E4M3 as the OCP 8-bit floating point format defines it: bit 7 the sign, bits 6-3 the
 * exponent e with bias 7, bits 2-0 the mantissa m; no infinities.
 *   e = 0:              (-1)^s * (m / 8) * 2^(1 - 7)   (subnormals; m = 0 is a signed zero)
 *   e = 15 and m = 7:   NaN
 *   otherwise:          (-1)^s * (1 + m / 8) * 2^(e - 7)
 */
static double e4m3_to_f64(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* attn_ref_e4m3_to_f64: decode n codes (for the pins). */
void attn_ref_e4m3_to_f64(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = e4m3_to_f64(codes[i]);
}

/*
 * attn_ref_rows_e4m3qk_f64: O and LSE of selected rows with Q and K given as E4M3 codes.
 *
 *   q8 [BH, Nq, d], k8 [BH, Nk, d]   E4M3 codes, C order
 *   v  [BH, Nk, dv]                  BF16 bit patterns
 *   q_descale, k_descale             the per-tensor factors of the real inputs
 * Other arguments and the return value as attn_ref_rows_f64.
 */
static int rows_e4m3qk(const uint8_t *q8, const uint8_t *k8, const uint16_t *v,
                       int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                       double scale, double q_descale, double k_descale,
                       const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads, int causal,
                       const uint16_t *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || nsel < 0 || (causal && Nq > Nk)) return REF_EINVAL;
    if (bias && (H < 1 || BH % H != 0 || sb < 0 || sh < 0 || sq < 0)) return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q8 || !k8 || !v || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                const uint8_t *qi = q8 + (bh * Nq + i) * d, *kh = k8 + bh * Nk * d;
                const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;   /* the row's keys */
                /* step 1 on the real inputs q_descale * Q8 and k_descale * K8 */
                for (int64_t j = 0; j < nk; j++) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; c++)
                        acc += (q_descale * e4m3_to_f64(qi[c])) * (k_descale * e4m3_to_f64(kh[j * d + c]));
                    s[j] = scale * acc;
                }
                if (bias) {   /* the optional B of the definition, one BF16 row per query */
                    const uint16_t *brow = bias + (bh / H) * sb + (bh % H) * sh + i * sq;
                    for (int64_t j = 0; j < nk; j++) s[j] += bf16_to_f64(brow[j]);
                }
                /* steps 2-5 with the head's BF16 value rows */
                const uint16_t *vrows = v + bh * Nk * dv;
                double *orow = o + r * dv;
                double mx = row_max(s, nk);
                double den = row_exp_sum(s, nk, mx);
                for (int64_t c = 0; c < dv; c++) {
                    double num = 0.0;
                    for (int64_t j = 0; j < nk; j++)
                        num += s[j] * bf16_to_f64(vrows[j * dv + c]);
                    orow[c] = num / den;
                }
                lse[r] = mx + log(den);
            }
            free(s);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

/*
 * attn_ref_rows_e4m3_f64: as attn_ref_rows_e4m3qk_f64 with V given as E4M3 codes too,
 * v8 [BH, Nk, dv] in C order with its descale factor: the real values are v_descale * V8,
 * and O is the definition's weighted sum of them (P is not rounded here).
 */
static int rows_e4m3(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                     int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                     double scale, double q_descale, double k_descale, double v_descale,
                     const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads, int causal,
                     const uint16_t *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || nsel < 0 || (causal && Nq > Nk)) return REF_EINVAL;
    if (bias && (H < 1 || BH % H != 0 || sb < 0 || sh < 0 || sq < 0)) return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q8 || !k8 || !v8 || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *w = (double *)malloc((size_t)Nk * sizeof(double));
        if (!w) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                const uint8_t *qrow = q8 + (bh * Nq + i) * d, *khead = k8 + bh * Nk * d, *vhead = v8 + bh * Nk * dv;
                const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;   /* the row's keys */
                /* step 1 on the real inputs */
                for (int64_t j = 0; j < nk; j++) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; c++)
                        dot += (q_descale * e4m3_to_f64(qrow[c])) * (k_descale * e4m3_to_f64(khead[j * d + c]));
                    w[j] = scale * dot;
                }
                if (bias) {   /* the optional B of the definition */
                    const uint16_t *bq = bias + (bh / H) * sb + (bh % H) * sh + i * sq;
                    for (int64_t j = 0; j < nk; j++) w[j] += bf16_to_f64(bq[j]);
                }
                /* steps 2-5 with the real values v_descale * V8 */
                double top = row_max(w, nk);
                double sum = row_exp_sum(w, nk, top);
                for (int64_t c = 0; c < dv; c++) {
                    double num = 0.0;
                    for (int64_t j = 0; j < nk; j++)
                        num += w[j] * (v_descale * e4m3_to_f64(vhead[j * dv + c]));
                    o[r * dv + c] = num / sum;
                }
                lse[r] = top + log(sum);
            }
            free(w);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

int attn_ref_rows_e4m3qk_f64(const uint8_t *q8, const uint8_t *k8, const uint16_t *v,
                             int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                             double scale, double q_descale, double k_descale,
                             const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_e4m3qk(q8, k8, v, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, sel, nsel, o, lse, nthreads, 0,
                       NULL, 1, 0, 0, 0);
}

int attn_ref_rows_e4m3_f64(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                           int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                           double scale, double q_descale, double k_descale, double v_descale,
                           const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_e4m3(q8, k8, v8, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, v_descale, sel, nsel, o, lse,
                     nthreads, 0, NULL, 1, 0, 0, 0);
}

/*
 * The two FP8 functions above under the causal mask of attn_ref_rows_causal_f64 (the
 * definition's optional mask B, "FlashAttention'ı Anlamak Bölüm 1", section 0.2, aligned to
 * the bottom-right corner): row i uses keys 0 .. i + (Nk - Nq) only, every sum running over
 * them. Requires Nq <= Nk.
 */
int attn_ref_rows_e4m3qk_causal_f64(const uint8_t *q8, const uint8_t *k8, const uint16_t *v,
                                    int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                                    double scale, double q_descale, double k_descale,
                                    const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_e4m3qk(q8, k8, v, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, sel, nsel, o, lse, nthreads, 1,
                       NULL, 1, 0, 0, 0);
}

int attn_ref_rows_e4m3_causal_f64(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                                  int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                                  double scale, double q_descale, double k_descale, double v_descale,
                                  const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_e4m3(q8, k8, v8, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, v_descale, sel, nsel, o, lse,
                     nthreads, 1, NULL, 1, 0, 0, 0);
}

/*
 * The two FP8 functions with the definition's optional additive bias B ("FlashAttention'ı
 * Anlamak Bölüm 1", section 0.2: S = QK^T / sqrt(d) + B) added to each score after the
 * scale, as attn_ref_rows_bias_f64 adds it: B_ij of head (b, h) = bias[b * sb + h * sh +
 * i * sq + j] (BF16 bits, strides in elements, 0 repeats), H heads per batch. -inf removes
 * a key; a row of only -inf has no softmax (NaN). No causal mask (the bias can carry one).
 */
int attn_ref_rows_e4m3qk_bias_f64(const uint8_t *q8, const uint8_t *k8, const uint16_t *v,
                                  const uint16_t *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq,
                                  int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                                  double scale, double q_descale, double k_descale,
                                  const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    if (!bias) return REF_EINVAL;
    return rows_e4m3qk(q8, k8, v, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, sel, nsel, o, lse, nthreads, 0,
                       bias, H, sb, sh, sq);
}

int attn_ref_rows_e4m3_bias_f64(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                                const uint16_t *bias, int64_t H, int64_t sb, int64_t sh, int64_t sq,
                                int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                                double scale, double q_descale, double k_descale, double v_descale,
                                const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    if (!bias) return REF_EINVAL;
    return rows_e4m3(q8, k8, v8, BH, Nq, Nk, d, dv, scale, q_descale, k_descale, v_descale, sel, nsel, o, lse,
                     nthreads, 0, bias, H, sb, sh, sq);
}

/*
 * MXFP8 inputs (the "MXFP8" of "Flash Attention на 5090 в CUDA C++", section "Что дальше").
 *
 * Read as the OCP microscaling format: E4M3 elements in blocks of 32 along the dimension a
 * product contracts over, each block with one E8M0 scale, an unsigned 8-bit exponent e
 * standing for 2^(e - 127) (e = 255 is NaN). The real inputs are
 *   q[i,c] = 2^(sq[i, c/32] - 127) * E4M3(q8[i,c])        blocks along d
 *   k[j,c] = 2^(sk[j, c/32] - 127) * E4M3(k8[j,c])        blocks along d
 *   v[j,c] = 2^(sv[j/32, c] - 127) * E4M3(v8[j,c])        blocks along the keys
 * and the definition is applied to them unchanged.
 */
static double e8m0_to_f64(uint8_t e)
{
    if (e == 255) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* attn_ref_e8m0_to_f64: decode n scale codes (for the pins). */
void attn_ref_e8m0_to_f64(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = e8m0_to_f64(codes[i]);
}

/*
 * attn_ref_rows_mxfp8_f64: O and LSE of selected rows from MXFP8 Q, K and V.
 *
 *   q8 [BH, Nq, d], k8 [BH, Nk, d], v8 [BH, Nk, dv]   E4M3 codes, C order
 *   sq [BH, Nq, d/32], sk [BH, Nk, d/32]              E8M0 scales of 32 elements along d
 *   sv [BH, ceil(Nk/32), dv]                          E8M0 scales of 32 keys per column
 * d must be a multiple of 32. Other arguments and the return value as attn_ref_rows_f64.
 */
static int rows_mxfp8(const uint8_t *q8, const uint8_t *sq, const uint8_t *k8, const uint8_t *sk,
                      const uint8_t *v8, const uint8_t *sv,
                      int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv, double scale,
                      const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads, int causal)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 32 || d % 32 != 0 || dv < 1 || nsel < 0 || (causal && Nq > Nk))
        return REF_EINVAL;
    if (nsel == 0) return REF_OK;
    if (!q8 || !sq || !k8 || !sk || !v8 || !sv || !sel || !o || !lse) return REF_EINVAL;
    for (int64_t r = 0; r < nsel; r++)
        if (sel[r] < 0 || sel[r] >= BH * Nq) return REF_EINVAL;
    const int64_t db = d / 32, kb = (Nk + 31) / 32;

    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#else
    (void)nthreads;
#endif
    {
        double *sc = (double *)malloc((size_t)Nk * sizeof(double));
        if (!sc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nsel; r++) {
                int64_t bh = sel[r] / Nq, i = sel[r] % Nq;
                const uint8_t *qi = q8 + (bh * Nq + i) * d, *qs = sq + (bh * Nq + i) * db;
                const uint8_t *kh = k8 + bh * Nk * d, *ks = sk + bh * Nk * db;
                const uint8_t *vh = v8 + bh * Nk * dv, *vs = sv + bh * kb * dv;
                const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;   /* the row's keys */
                /* step 1 on the real inputs */
                for (int64_t j = 0; j < nk; j++) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; c++)
                        dot += (e8m0_to_f64(qs[c / 32]) * e4m3_to_f64(qi[c])) *
                               (e8m0_to_f64(ks[j * db + c / 32]) * e4m3_to_f64(kh[j * d + c]));
                    sc[j] = scale * dot;
                }
                /* steps 2-5 with the real values */
                double top = row_max(sc, nk);
                double den = row_exp_sum(sc, nk, top);
                for (int64_t c = 0; c < dv; c++) {
                    double num = 0.0;
                    for (int64_t j = 0; j < nk; j++)
                        num += sc[j] * (e8m0_to_f64(vs[(j / 32) * dv + c]) * e4m3_to_f64(vh[j * dv + c]));
                    o[r * dv + c] = num / den;
                }
                lse[r] = top + log(den);
            }
            free(sc);
        }
    }
    return failed ? REF_ENOMEM : REF_OK;
}

int attn_ref_rows_mxfp8_f64(const uint8_t *q8, const uint8_t *sq, const uint8_t *k8, const uint8_t *sk,
                            const uint8_t *v8, const uint8_t *sv,
                            int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv, double scale,
                            const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_mxfp8(q8, sq, k8, sk, v8, sv, BH, Nq, Nk, d, dv, scale, sel, nsel, o, lse, nthreads, 0);
}

/*
 * attn_ref_rows_mxfp8_causal_f64: attn_ref_rows_mxfp8_f64 under the causal mask of
 * attn_ref_rows_causal_f64 (row i uses keys 0 .. i + (Nk - Nq) only; needs Nq <= Nk).
 */
int attn_ref_rows_mxfp8_causal_f64(const uint8_t *q8, const uint8_t *sq, const uint8_t *k8, const uint8_t *sk,
                                   const uint8_t *v8, const uint8_t *sv,
                                   int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv, double scale,
                                   const int64_t *sel, int64_t nsel, double *o, double *lse, int nthreads)
{
    return rows_mxfp8(q8, sq, k8, sk, v8, sv, BH, Nq, Nk, d, dv, scale, sel, nsel, o, lse, nthreads, 1);
}
