/*
 * fa2_oracle.c -- plain, slow, fp64 CPU oracle for exact scaled-dot-product
 * attention with per-row logsumexp.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load or call this code.  The
 * product path (the CUDA library) never routes through it and shares no code,
 * header, table or helper with it.
 *
 * What it computes (the textbook definition the FlashAttention pages state and
 * that the tiled method reproduces exactly, up to rounding):
 *
 *   - Olowookere, "FlashAttention-2 from scratch with a custom Triton kernel",
 *     section "The core idea: making attention IO-aware":
 *         S = Q K^T,  P = softmax(S) (row-wise),  O = P V.
 *   - "Flash Attention: principles and implementation" (tbr8.org), section 1
 *     ("the compute bottleneck of attention"): softmax(Q K^T / sqrt(d)) V,
 *     i.e. the scores carry the scale factor before the softmax.
 *   - "Chapter 08: Flash Attention -- blocked attention" (chuoer47), section 3
 *     ("LSE"): the per-row log-sum-exp LSE = m + log(l) is what a backward
 *     pass needs; section 4 ("causal mask"): query i may see key j only when
 *     j <= i (lower triangle including the diagonal).
 *
 * Readings taken where the pages are loose:
 *   - LSE is the NATURAL log of sum_j exp(s_ij) over the SCALED scores
 *     s_ij = scale * q_i . k_j (the plain definition; page 4's base-2 value is
 *     this times log2(e)).
 *   - Masked positions are excluded exactly (weight 0), not given -1e6.
 *   - Causal with Lq != Lk uses the literal top-left rule j <= i.
 *   - Keys j >= Lk do not exist (no zero-padded keys take part).
 *
 * Per output row (b, h, i) the oracle MATERIALISES the full score row
 * S[i, 0..Lk) and the full probability row P[i, 0..Lk) in fp64 before any
 * reduction; there is no tiling, no online softmax, no fusion.
 *
 * Inputs are bf16 bit patterns (uint16) in contiguous (B, H, L, D) order; each
 * is widened exactly to fp64 (bf16 is the top half of an IEEE binary32).
 * Parallelism is over independent output rows only (OpenMP), which does not
 * change any row's arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64, exact: the 16 bits are the high half of a binary32. */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exposed so a test can pin the widening against an independent decoder. */
void fa2_oracle_decode_bf16(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = bf16_to_f64(src[t]);
}

/*
 * Key j is visible to query i: the causal mask of chapter 08, section 4 (j <= i),
 * and, with window >= 0, the sliding window of "Flash Attention: principles and
 * implementation" (tbr8.org), section 6.3 -- window_size = (w, 0) with causal:
 * w keys to the left of the query and none to the right, i.e. i - w <= j <= i.
 */
static int allowed(int64_t i, int64_t j, int causal, int64_t window)
{
    return (!causal || j <= i) && (window < 0 || j >= i - window);
}

/*
 * One output row.  s and p are caller-provided scratch rows of length Lk.
 * Returns the number of visible keys |A_i|.
 */
static int64_t one_row(const uint16_t *q_row, const uint16_t *k_head,
                       const uint16_t *v_head, int64_t i, int64_t Lk,
                       int64_t D, int causal, int64_t window, double scale, double *s,
                       double *p, double *o_row, double *lse_out)
{
    /* S row: s_j = scale * sum_d q_id k_jd  (fp64, inputs widened exactly). */
    int64_t n_allowed = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < Lk; ++j) {
        if (!allowed(i, j, causal, window)) {
            s[j] = -INFINITY; /* not in A_i; never read below */
            continue;
        }
        const uint16_t *k_row = k_head + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += bf16_to_f64(q_row[d]) * bf16_to_f64(k_row[d]);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
        ++n_allowed;
    }

    /* P row: p_j = exp(s_j - M) / sum_{A_i} exp(s_j - M);  p_j = 0 off A_i. */
    double z = 0.0;
    for (int64_t j = 0; j < Lk; ++j) {
        if (allowed(i, j, causal, window)) {
            p[j] = exp(s[j] - m);
            z += p[j];
        } else {
            p[j] = 0.0;
        }
    }
    for (int64_t j = 0; j < Lk; ++j)
        p[j] = p[j] / z;

    /* O row: o_d = sum_j p_j v_jd. */
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = 0.0;
    for (int64_t j = 0; j < Lk; ++j) {
        if (!allowed(i, j, causal, window))
            continue;
        const uint16_t *v_row = v_head + j * D;
        for (int64_t d = 0; d < D; ++d)
            o_row[d] += p[j] * bf16_to_f64(v_row[d]);
    }

    /* LSE_i = M + ln sum_{A_i} exp(s_j - M)  (= ln sum exp(s_j)). */
    *lse_out = m + log(z);
    return n_allowed;
}

/*
 * Attention for a list of output rows.
 *
 *   q: bf16 bits (B, H, Lq, D);  k, v: bf16 bits (B, H, Lk, D); contiguous.
 *   rows[r] = (b * H + h) * Lq + i selects output row r.
 *   o:   fp64 (n_rows, D), lse: fp64 (n_rows).
 *   p_out: optional fp64 (n_rows, Lk) copy of the materialised P rows.
 *   n_threads <= 0 lets OpenMP choose.
 *
 * Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 */
int fa2_oracle_rows_w(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t D,
                      int causal, int64_t window, double scale, const int64_t *rows,
                      int64_t n_rows, double *o, double *lse, double *p_out,
                      int n_threads)
{
    if (!q || !k || !v || !o || !lse || (n_rows > 0 && !rows))
        return 1;
    if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0 || n_rows < 0)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * Lq)
            return 1;

    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Lk * sizeof(double));
        double *p = (double *)malloc((size_t)Lk * sizeof(double));
        if (!s || !p) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t bh = rows[r] / Lq;
                int64_t i = rows[r] % Lq;
                const uint16_t *q_row = q + (bh * Lq + i) * D;
                const uint16_t *k_head = k + bh * Lk * D;
                const uint16_t *v_head = v + bh * Lk * D;
                one_row(q_row, k_head, v_head, i, Lk, D, causal, window, scale, s, p,
                        o + r * D, lse + r);
                if (p_out)
                    memcpy(p_out + r * Lk, p, (size_t)Lk * sizeof(double));
            }
        }
        free(s);
        free(p);
    }
    return failed ? 2 : 0;
}

/*
 * ------------------------------------------------------------------ gradients
 *
 * The backward pass of the same attention ("Chapter 08: Flash Attention --
 * blocked attention", section 6: 6.2 the per-row scalar Delta, 6.3 the softmax
 * backward, 6.4 the three gradient lines).  Given the upstream gradient dO of a
 * loss L with respect to O, the gradients of L with respect to the inputs are,
 * per (b, h), with P the materialised probabilities of the forward definition:
 *
 *   Delta_i = sum_d dO_id * O_id                       (one scalar per query row)
 *   dP_ij   = sum_d dO_id * V_jd                       (dP = dO V^T)
 *   dS_ij   = P_ij * (dP_ij - Delta_i)                 (softmax backward; dS is the
 *                                                       gradient of the scaled score)
 *   dV_jd   = sum_i P_ij * dO_id                       (dV = P^T dO)
 *   dK_jd   = scale * sum_i dS_ij * Q_id               (dK = scale * dS^T Q)
 *   dQ_id   = scale * sum_j dS_ij * K_jd               (dQ = scale * dS K)
 *
 * Masked positions have P_ij = 0 and so contribute nothing.  The section works
 * in base 2 (P = 2^(S' - LSE_2) with S' carrying scale * log2 e, hence its ln 2
 * factors); in natural-log terms with the scale applied to the scores the
 * factors cancel into the plain expressions above.
 *
 * Per query row the oracle materialises the full P row (through one_row, the
 * forward definition), the full dP row and the full dS row in fp64 before
 * using them, and accumulates dK, dV over the rows in row order (one head per
 * thread, so the order is fixed).
 */

/* fp64 forward for fp64 inputs (contiguous (B, H, L, D)); same row definition. */
static int64_t one_row_f64(const double *q_row, const double *k_head, const double *v_head, int64_t i,
                           int64_t Lk, int64_t D, int causal, int64_t window, double scale, double *s, double *p,
                           double *o_row, double *lse_out)
{
    int64_t n_allowed = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < Lk; ++j) {
        if (!allowed(i, j, causal, window)) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += q_row[d] * k_head[j * D + d];
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
        ++n_allowed;
    }
    double z = 0.0;
    for (int64_t j = 0; j < Lk; ++j) {
        if (allowed(i, j, causal, window)) {
            p[j] = exp(s[j] - m);
            z += p[j];
        } else {
            p[j] = 0.0;
        }
    }
    for (int64_t j = 0; j < Lk; ++j)
        p[j] = p[j] / z;
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = 0.0;
    for (int64_t j = 0; j < Lk; ++j) {
        if (!allowed(i, j, causal, window))
            continue;
        for (int64_t d = 0; d < D; ++d)
            o_row[d] += p[j] * v_head[j * D + d];
    }
    *lse_out = m + log(z);
    return n_allowed;
}

/*
 * Forward for fp64 inputs, every row: o (B, H, Lq, D), lse (B, H, Lq).  Lets a
 * test differentiate the forward definition numerically.  Returns as
 * fa2_oracle_rows.
 */
int fa2_oracle_fwd_f64(const double *q, const double *k, const double *v, int64_t B, int64_t H, int64_t Lq,
                       int64_t Lk, int64_t D, int causal, int64_t window, double scale, double *o, double *lse,
                       int n_threads)
{
    if (!q || !k || !v || !o || !lse || B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0)
        return 1;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Lk * sizeof(double));
        double *p = (double *)malloc((size_t)Lk * sizeof(double));
        if (!s || !p) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < B * H * Lq; ++r) {
                const int64_t bh = r / Lq, i = r % Lq;
                one_row_f64(q + r * D, k + bh * Lk * D, v + bh * Lk * D, i, Lk, D, causal, window, scale, s, p,
                            o + r * D, lse + r);
            }
        }
        free(s);
        free(p);
    }
    return failed ? 2 : 0;
}

/* Gradients of one head (all fp64); s, p, dp: scratch rows of Lk; o_row: D. */
static void one_head_bwd(const double *q, const double *k, const double *v, const double *dout, int64_t Lq,
                         int64_t Lk, int64_t D, int causal, int64_t window, double scale, double *dq, double *dk,
                         double *dv, double *delta, double *s, double *p, double *dp, double *o_row)
{
    for (int64_t t = 0; t < Lk * D; ++t) {
        dk[t] = 0.0;
        dv[t] = 0.0;
    }
    for (int64_t i = 0; i < Lq; ++i) {
        const double *q_row = q + i * D, *do_row = dout + i * D;
        double lse;
        one_row_f64(q_row, k, v, i, Lk, D, causal, window, scale, s, p, o_row, &lse);
        /* Delta_i = dO_i . O_i */
        double dl = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dl += do_row[d] * o_row[d];
        if (delta)
            delta[i] = dl;
        /* dP row, then dS row (kept in dp) */
        for (int64_t j = 0; j < Lk; ++j) {
            if (!allowed(i, j, causal, window)) {
                dp[j] = 0.0;
                continue;
            }
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += do_row[d] * v[j * D + d];
            dp[j] = p[j] * (acc - dl);
        }
        /* dQ_i = scale * sum_j dS_ij K_j;  dK_j += scale * dS_ij Q_i;  dV_j += P_ij dO_i */
        double *dq_row = dq + i * D;
        for (int64_t d = 0; d < D; ++d)
            dq_row[d] = 0.0;
        for (int64_t j = 0; j < Lk; ++j) {
            if (!allowed(i, j, causal, window))
                continue;
            for (int64_t d = 0; d < D; ++d) {
                dq_row[d] += dp[j] * k[j * D + d];
                dk[j * D + d] += dp[j] * q_row[d];
                dv[j * D + d] += p[j] * do_row[d];
            }
        }
        for (int64_t d = 0; d < D; ++d)
            dq_row[d] *= scale;
    }
    for (int64_t t = 0; t < Lk * D; ++t)
        dk[t] *= scale;
}

/*
 * Gradients for fp64 inputs, every head: dq (B, H, Lq, D), dk and dv (B, H, Lk,
 * D); delta (B, H, Lq) optional.  Returns as fa2_oracle_rows.
 */
int fa2_oracle_bwd_f64(const double *q, const double *k, const double *v, const double *dout, int64_t B,
                       int64_t H, int64_t Lq, int64_t Lk, int64_t D, int causal, int64_t window, double scale,
                       double *dq, double *dk, double *dv, double *delta, int n_threads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0)
        return 1;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Lk * sizeof(double));
        double *p = (double *)malloc((size_t)Lk * sizeof(double));
        double *dp = (double *)malloc((size_t)Lk * sizeof(double));
        double *o_row = (double *)malloc((size_t)D * sizeof(double));
        if (!s || !p || !dp || !o_row) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < B * H; ++bh)
                one_head_bwd(q + bh * Lq * D, k + bh * Lk * D, v + bh * Lk * D, dout + bh * Lq * D, Lq, Lk, D,
                             causal, window, scale, dq + bh * Lq * D, dk + bh * Lk * D, dv + bh * Lk * D,
                             delta ? delta + bh * Lq : NULL, s, p, dp, o_row);
        }
        free(s);
        free(p);
        free(dp);
        free(o_row);
    }
    return failed ? 2 : 0;
}

/*
 * ------------------------------------------------------------------ FP8 inputs
 *
 * The FP8 forward that "Flash Attention: principles and implementation"
 * (tbr8.org), section 4.3, names for FlashAttention-3 without fixing a format.
 * Reading taken: Q, K and V are stored as e4m3 (1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities, exponent 15 with mantissa 7 is NaN;
 * largest finite value 448), each with one fp32 descale factor per (batch, head):
 * the real input is the stored value times its descale.  The oracle widens the
 * stored values exactly, multiplies by the descale in fp64 (exact: at most 4 + 24
 * significant bits), and applies the attention definition above unchanged.
 */
static double e4m3_to_f64(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 3) & 0xF, m = bits & 0x7;
    if (e == 15 && m == 7)
        return NAN;
    /* subnormal (e = 0): m/8 * 2^-6;  normal: (1 + m/8) * 2^(e - 7) */
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + (double)m, e - 10);
    return sign ? -mag : mag;
}

/* Exposed so a test can pin the widening against an independent decoder. */
void fa2_oracle_decode_e4m3(const uint8_t *src, double *dst, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = e4m3_to_f64(src[t]);
}

/*
 * Real values of an e4m3 tensor (BH heads of `per_head` elements, contiguous):
 * out[h][e] = e4m3(x[h][e]) * descale[h].
 */
void fa2_oracle_dequant_e4m3(const uint8_t *x, const float *descale, int64_t BH, int64_t per_head, double *out)
{
    for (int64_t h = 0; h < BH; ++h)
        for (int64_t e = 0; e < per_head; ++e)
            out[h * per_head + e] = e4m3_to_f64(x[h * per_head + e]) * (double)descale[h];
}

/*
 * Attention for a list of output rows of fp64 inputs (contiguous (B, H, L, D)):
 * the same row definition as fa2_oracle_rows_w.  Returns as fa2_oracle_rows_w.
 */
int fa2_oracle_rows_f64(const double *q, const double *k, const double *v, int64_t B, int64_t H, int64_t Lq,
                        int64_t Lk, int64_t D, int causal, int64_t window, double scale, const int64_t *rows,
                        int64_t n_rows, double *o, double *lse, int n_threads)
{
    if (!q || !k || !v || !o || !lse || (n_rows > 0 && !rows))
        return 1;
    if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0 || n_rows < 0)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * Lq)
            return 1;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Lk * sizeof(double));
        double *p = (double *)malloc((size_t)Lk * sizeof(double));
        if (!s || !p) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < n_rows; ++r) {
                const int64_t bh = rows[r] / Lq, i = rows[r] % Lq;
                one_row_f64(q + rows[r] * D, k + bh * Lk * D, v + bh * Lk * D, i, Lk, D, causal, window, scale,
                            s, p, o + r * D, lse + r);
            }
        }
        free(s);
        free(p);
    }
    return failed ? 2 : 0;
}

/* fa2_oracle_rows_w without a window. */
int fa2_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t D,
                    int causal, double scale, const int64_t *rows,
                    int64_t n_rows, double *o, double *lse, double *p_out,
                    int n_threads)
{
    return fa2_oracle_rows_w(q, k, v, B, H, Lq, Lk, D, causal, -1, scale, rows, n_rows, o, lse, p_out,
                             n_threads);
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int fa2_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
