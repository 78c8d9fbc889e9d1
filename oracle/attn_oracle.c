/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for the dense attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * What it computes (the plain definition the method reaches up to rounding):
 *   "B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams",
 *   Chapter 1 section ii (work decomposition over [B, H, S, D] tensors) and
 *   section B (online softmax: the tiled loop must reproduce ordinary softmax);
 *   "Learning FlashAttention the Hard Way, Part 2", Move 0 (scores, a max pass,
 *   a sum-of-exponentials pass, then the weighted sum of V rows);
 *   "Attention for sm90, Line by Line", the exp2 question (the log-sum-exp
 *   residual is stored in natural-log units).
 *
 * For every batch b, head h and query row i, with the BF16 inputs widened
 * exactly to fp64:
 *     s_ij   = scale * sum_d q_id * k_jd
 *     m_i    = max_j s_ij
 *     l_i    = sum_j exp(s_ij - m_i)
 *     o_id   = (sum_j exp(s_ij - m_i) * v_jd) / l_i
 *     lse_i  = m_i + ln(l_i)
 * The score row is materialised (Sk doubles), then traversed three times, as
 * in the two-kernel scalar formulation.  No blocking, no online rescaling.
 *
 * causal != 0 restricts row i to keys j <= i (top-left aligned: query i and
 * key i share a position, as torch.nn.functional.scaled_dot_product_attention
 * with is_causal=True does); every row keeps at least key 0.  The pages name
 * causal masking for the sm90 kernel ("Attention for sm90, Line by Line", the
 * persistent-flag question) without fixing an alignment; top-left is the plain
 * reading for Sq == Sk and keeps every row non-empty for any Sq, Sk.
 *
 * Layout: q [B,H,Sq,D], k and v [B,H,Sk,D], all contiguous BF16 bit patterns
 * (uint16).  o [B,H,Sq,D] fp64, lse [B,H,Sq] fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* A BF16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row of one (b, h): materialised two-pass softmax. */
static void oracle_row(const uint16_t *q_row, const uint16_t *k_head, const uint16_t *v_head,
                       int64_t Sk, int64_t D, double scale,
                       double *s, double *o_row, double *lse_out)
{
    /* Sk here is the number of keys this row attends (all keys, or i + 1 when causal). */
    for (int64_t j = 0; j < Sk; ++j) {
        const uint16_t *k_row = k_head + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += bf16_to_f64(q_row[d]) * bf16_to_f64(k_row[d]);
        s[j] = scale * dot;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < Sk; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < Sk; ++j)
        l += exp(s[j] - m);
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = 0.0;
    for (int64_t j = 0; j < Sk; ++j) {
        const double p = exp(s[j] - m);
        const uint16_t *v_row = v_head + j * D;
        for (int64_t d = 0; d < D; ++d)
            o_row[d] += p * bf16_to_f64(v_row[d]);
    }
    for (int64_t d = 0; d < D; ++d)
        o_row[d] /= l;
    *lse_out = m + log(l);
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_max_threads(void) { return set_threads(0); }

/* Keys attended by query row i. */
static int64_t keys_for_row(int64_t i, int64_t Sk, int causal)
{
    if (!causal) return Sk;
    return i + 1 < Sk ? i + 1 : Sk;
}

/*
 * Full forward.  Returns 0 on success, -1 on a bad argument, -2 when the
 * per-thread score buffer cannot be allocated.
 */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D,
                    double scale, int causal, double *o, double *lse, int nthreads)
{
    if (B < 0 || H < 0 || Sq < 0 || Sk <= 0 || D <= 0) return -1;
    set_threads(nthreads);
    const int64_t rows = B * H * Sq;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Sk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!s) continue;
            const int64_t bh = r / Sq;
            oracle_row(q + r * D, k + bh * Sk * D, v + bh * Sk * D,
                       keys_for_row(r - bh * Sq, Sk, causal), D, scale, s, o + r * D, lse + r);
        }
        free(s);
    }
    return err;
}

/*
 * Selected rows only: row n of the output is query row row_idx[n] of the
 * flattened head bh_idx[n] (bh = b*H + h).  o_rows is [nrows, D], lse_rows is
 * [nrows].  Used to check sampled outputs of full-size problems.
 */
int oracle_attn_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D,
                         double scale, int causal, const int64_t *bh_idx, const int64_t *row_idx,
                         int64_t nrows, double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || H < 0 || Sq < 0 || Sk <= 0 || D <= 0 || nrows < 0) return -1;
    for (int64_t n = 0; n < nrows; ++n)
        if (bh_idx[n] < 0 || bh_idx[n] >= B * H || row_idx[n] < 0 || row_idx[n] >= Sq)
            return -1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Sk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t n = 0; n < nrows; ++n) {
            if (!s) continue;
            const int64_t bh = bh_idx[n];
            oracle_row(q + (bh * Sq + row_idx[n]) * D, k + bh * Sk * D, v + bh * Sk * D,
                       keys_for_row(row_idx[n], Sk, causal), D, scale, s, o_rows + n * D,
                       lse_rows + n);
        }
        free(s);
    }
    return err;
}

/*
 * Materialised probabilities P = softmax(scale * Q K^T) for one head,
 * p [Sq, Sk] (entries of masked keys are 0).  For small shapes only.
 */
int oracle_attn_probs(const uint16_t *q_head, const uint16_t *k_head,
                      int64_t Sq, int64_t Sk, int64_t D, double scale, int causal, double *p)
{
    if (Sq < 0 || Sk <= 0 || D <= 0) return -1;
    for (int64_t i = 0; i < Sq; ++i) {
        double *s = p + i * Sk;
        const int64_t nk = keys_for_row(i, Sk, causal);
        for (int64_t j = nk; j < Sk; ++j) s[j] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dot += bf16_to_f64(q_head[i * D + d]) * bf16_to_f64(k_head[j * D + d]);
            s[j] = scale * dot;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j)
            if (s[j] > m) m = s[j];
        double l = 0.0;
        for (int64_t j = 0; j < nk; ++j)
            l += exp(s[j] - m);
        for (int64_t j = 0; j < nk; ++j)
            s[j] = exp(s[j] - m) / l;
    }
    return 0;
}

/*
 * Backward of the same plain definition, for one loss L with dL/dO = dO given:
 *     P     = softmax(scale * Q K^T)            (masked entries 0 when causal)
 *     dV    = P^T dO
 *     dP    = dO V^T
 *     dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik)
 *     dQ    = scale * dS K
 *     dK    = scale * dS^T Q
 * (the chain rule through O = P V and the softmax Jacobian; "Attention for
 * sm90, Line by Line", the exp2 question, is where the pages make the LSE the
 * forward's residual for this pass).  Row by row in fp64: p and dp of a query
 * row are materialised (Sk doubles each), dQ_i is finished per row, dK and dV
 * accumulate over rows.  Parallel over (b, h) only (dK/dV sum over rows).
 * do_ is [B,H,Sq,D] BF16 bits; dq [B,H,Sq,D], dk and dv [B,H,Sk,D] fp64.
 */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *do_,
                    int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D, double scale,
                    int causal, double *dq, double *dk, double *dv, int nthreads)
{
    if (B < 0 || H < 0 || Sq < 0 || Sk <= 0 || D <= 0) return -1;
    set_threads(nthreads);
    const int64_t heads = B * H;
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc((size_t)Sk * sizeof(double));
        double *dp = (double *)malloc((size_t)Sk * sizeof(double));
        if (!p || !dp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < heads; ++bh) {
            if (!p || !dp) continue;
            const uint16_t *qh = q + bh * Sq * D, *kh = k + bh * Sk * D, *vh = v + bh * Sk * D;
            const uint16_t *doh = do_ + bh * Sq * D;
            double *dqh = dq + bh * Sq * D, *dkh = dk + bh * Sk * D, *dvh = dv + bh * Sk * D;
            for (int64_t x = 0; x < Sk * D; ++x) { dkh[x] = 0.0; dvh[x] = 0.0; }
            for (int64_t i = 0; i < Sq; ++i) {
                const int64_t nk = keys_for_row(i, Sk, causal);
                /* p_i: softmax of the scaled scores of row i */
                double m = -INFINITY;
                for (int64_t j = 0; j < nk; ++j) {
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += bf16_to_f64(qh[i * D + d]) * bf16_to_f64(kh[j * D + d]);
                    p[j] = scale * dot;
                    if (p[j] > m) m = p[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < nk; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
                for (int64_t j = 0; j < nk; ++j) p[j] /= l;
                /* dp_i = dO_i V^T, delta_i = sum_j p_ij dp_ij */
                double delta = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += bf16_to_f64(doh[i * D + d]) * bf16_to_f64(vh[j * D + d]);
                    dp[j] = dot;
                    delta += p[j] * dot;
                }
                for (int64_t d = 0; d < D; ++d) dqh[i * D + d] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    const double ds = p[j] * (dp[j] - delta);
                    for (int64_t d = 0; d < D; ++d) {
                        dqh[i * D + d] += scale * ds * bf16_to_f64(kh[j * D + d]);
                        dkh[j * D + d] += scale * ds * bf16_to_f64(qh[i * D + d]);
                        dvh[j * D + d] += p[j] * bf16_to_f64(doh[i * D + d]);
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return err;
}
