/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of exact attention and of its gradient.
 * It exists to check the CUDA library; nothing in the product links it, and
 * it shares no code, header, table or constant with the CUDA path.
 * Only the tests, the package smoke check and the bench's CPU baseline use it.
 *
 * What it computes, row by row, straight from the definition (no tiling,
 * no online softmax, no reordering):
 *
 *   kv head      g   = h / (Hq / Hkv)   (contiguous groups of query heads
 *                                        share one key/value head)
 *   key set      J_i = {0..N-1}, or {0..i} when causal (key j is kept
 *                      for query i iff j <= i, diagonal included); with a
 *                      sliding window of W keys, J_i = {max(0, i-W+1)..i}
 *                      (key j kept iff i - W < j <= i)
 *   logit        s_ij = scale * sum_d q[i,d] k[j,d]  (+ bias[i,j])
 *   row max      m_i  = max_{j in J_i} s_ij
 *   row sum      l_i  = sum_{j in J_i} exp(s_ij - m_i)
 *   probability  P_ij = exp(s_ij - m_i) / l_i
 *   output       O_i  = sum_{j in J_i} P_ij v_j
 *   log-sum-exp  LSE_i = m_i + ln(l_i)
 *
 * Sources (cited by page title and section):
 *  - "FlashAttention原理与Triton实战：突破Attention显存瓶颈", section 2.1:
 *    standard attention S = QK^T, P = softmax(S), O = PV, S and P materialised.
 *  - kwkr.cn/news/592482 (FlashAttention tutorial), section 1.1: the scale
 *    1/sqrt(d) on QK^T; section 2.1: the two-pass safe softmax
 *    m = max, l = sum exp(s - m), P = exp(s - m) / l; section 3.4: the
 *    causal mask hides the strict upper triangle (triu, diagonal = 1).
 *  - blog.ans20xx.com/posts/ai/day26, "最小 attention wrapper": the naive
 *    attention with a lower-triangular (tril) keep mask and scale d^-0.5.
 *  - Sliding-window (local) attention: "FlashAttention原理与Triton实战",
 *    sections 3.1 and 7 (a window mask stacked on the causal kernel) and the
 *    Block Attention Residual page, "实验结果" (an SWA baseline).  The pages
 *    give no formula; the window here is the causal one over the W most
 *    recent keys, the query's own key included.
 *  - Block Attention Residual Triton kernel (iqiancheng.github.io), section
 *    "Block Attention Residual 做了什么": softmax(Q_i K_i^T / sqrt(d) +
 *    logit_residual_{i-1}); the residual is added unscaled to the scaled
 *    logits, and the emitted logits are the sum before the softmax.
 *  - Backward by recomputation from the saved per-row statistics:
 *    kwkr.cn/news/592482 section 2.4 and "FlashAttention原理与Triton实战"
 *    sections 2.3 and 4.3 (dS subtracts a row sum). The gradient below is the
 *    exact derivative of the forward definition:
 *      P_ij   = exp(s_ij - LSE_i)
 *      dV_j   = sum_i P_ij dO_i
 *      dP_ij  = dO_i . v_j
 *      Delta_i = sum_d dO_i[d] O_i[d]            (= sum_j P_ij dP_ij)
 *      dS_ij  = P_ij (dP_ij - Delta_i)
 *      dQ_i   = scale * sum_j dS_ij k_j
 *      dK_j   = scale * sum_i dS_ij q_i
 *    For grouped heads, dK and dV of a kv head sum over its query heads.
 *
 * Data: q [B,Hq,N,D], k and v [B,Hkv,N,D] (and dO like q) as double (the
 * bf16 inputs widen exactly), bias [B,Hq,N,N] as double or NULL. All
 * arithmetic is double.
 * Rows are addressed by their flat index r = (b*Hq + h)*N + i; key rows by
 * (b*Hkv + g)*N + j. Outputs are written per requested row, in request order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads used by the parallel loops (rows are independent). */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* J_i as the half-open key range [*j0, *j1); window <= 0 means none. */
static void key_range(int64_t i, int64_t N, int causal, int64_t window, int64_t *j0, int64_t *j1)
{
    *j1 = causal ? i + 1 : N;
    *j0 = (causal && window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
}

/* s_ij for every j in J_i of one query row, written to s[0..|J_i|). */
static void row_logits(const double *q_row, const double *k_head, const double *bias_row,
                       int64_t nk, int64_t D, double scale, double *s)
{
    for (int64_t j = 0; j < nk; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += q_row[d] * k_head[j * D + d];
        s[j] = scale * dot + (bias_row ? bias_row[j] : 0.0);
    }
}

/* Two-pass softmax statistics of one row: m = max s, l = sum exp(s - m). */
static void row_stats(const double *s, int64_t nk, double *m_out, double *l_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < nk; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j)
        l += exp(s[j] - m);
    *m_out = m;
    *l_out = l;
}

/*
 * Forward pass for the listed query rows.
 *   o      [nrows, D]  output rows O_i
 *   lse    [nrows]     LSE_i = m_i + ln l_i (may be NULL)
 *   logits [nrows, N]  s_ij for j in J_i; other entries left as they were
 *                      (may be NULL). May alias bias when the bias rows are
 *                      read in request order (each row reads its bias before
 *                      writing its logits).
 * rows == NULL means every row, in natural order.  bias is [B,Hq,N,N]
 * indexed by the flat row, or, when bias_per_request is nonzero, [nrows, N]
 * indexed by request (the bias rows of the requested rows only).
 */
void orc_fwd_rows(const double *q, const double *k, const double *v, const double *bias,
                  int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t D,
                  double scale, int causal, int64_t window, const int64_t *rows,
                  int64_t nrows, int bias_per_request, double *o, double *lse, double *logits)
{
    (void)B;
    const int64_t group = Hq / Hkv;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            const int64_t i = flat % N;
            const int64_t bh = flat / N;
            const int64_t b = bh / Hq, h = bh % Hq;
            const int64_t g = h / group;
            const double *q_row = q + flat * D;
            const double *k_head = k + (b * Hkv + g) * N * D;
            const double *v_head = v + (b * Hkv + g) * N * D;
            const double *bias_row = bias ? bias + (bias_per_request ? r : flat) * N : NULL;
            int64_t j0, j1;
            key_range(i, N, causal, window, &j0, &j1);
            const int64_t nk = j1 - j0;   /* s[t] is the logit of key j0 + t */

            row_logits(q_row, k_head + j0 * D, bias_row ? bias_row + j0 : NULL, nk, D, scale, s);
            double m, l;
            row_stats(s, nk, &m, &l);

            double *o_row = o + r * D;
            for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
            for (int64_t t = 0; t < nk; ++t) {
                const double p = exp(s[t] - m) / l;
                for (int64_t d = 0; d < D; ++d)
                    o_row[d] += p * v_head[(j0 + t) * D + d];
            }
            if (lse) lse[r] = m + log(l);
            if (logits) {
                double *out = logits + r * N;
                for (int64_t t = 0; t < nk; ++t) out[j0 + t] = s[t];
            }
        }
        free(s);
    }
}

/*
 * Delta_i = sum_d dO_i[d] * O_i[d] for the listed rows.
 *   o [nrows, D] rows of O in request order; delta [nrows].
 */
void orc_delta_rows(const double *dO, const double *o, int64_t D,
                    const int64_t *rows, int64_t nrows, double *delta)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t flat = rows ? rows[r] : r;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d)
            acc += dO[flat * D + d] * o[r * D + d];
        delta[r] = acc;
    }
}

/*
 * dQ for the listed query rows.
 *   lse, delta: full [B,Hq,N] arrays, read at the listed rows only.
 *   bias:    [B,Hq,N,N] or NULL, the additive logit bias of the forward.
 *   grad_in: [B,Hq,N,N] or NULL, the gradient flowing into this layer's
 *            logits from the next layer of a block residual chain (the next
 *            layer adds these logits to its own, unscaled, so its total
 *            logit gradient arrives here unchanged).
 *   dq [nrows, D];  grad_out [nrows, N] or NULL: the total logit gradient
 *   dS_ij for j in J_i (also the gradient of the loss w.r.t. bias_ij),
 *   0 for the keys outside J_i.
 * With both NULL this is the plain attention backward.
 */
void orc_bwd_dq_rows(const double *q, const double *k, const double *v, const double *dO,
                     const double *lse, const double *delta, const double *bias,
                     const double *grad_in,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t D,
                     double scale, int causal, int64_t window, const int64_t *rows,
                     int64_t nrows, double *dq, double *grad_out)
{
    (void)B;
    const int64_t group = Hq / Hkv;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            const int64_t i = flat % N;
            const int64_t bh = flat / N;
            const int64_t b = bh / Hq, h = bh % Hq;
            const int64_t g = h / group;
            const double *k_head = k + (b * Hkv + g) * N * D;
            const double *v_head = v + (b * Hkv + g) * N * D;
            const double *do_row = dO + flat * D;
            int64_t j0, j1;
            key_range(i, N, causal, window, &j0, &j1);
            const int64_t nk = j1 - j0;

            row_logits(q + flat * D, k_head + j0 * D, bias ? bias + flat * N + j0 : NULL, nk, D,
                       scale, s);
            double *dq_row = dq + r * D;
            for (int64_t d = 0; d < D; ++d) dq_row[d] = 0.0;
            double *go = grad_out ? grad_out + r * N : NULL;
            if (go)
                for (int64_t j = 0; j < N; ++j) go[j] = 0.0;
            for (int64_t t = 0; t < nk; ++t) {
                const int64_t j = j0 + t;
                const double p = exp(s[t] - lse[flat]);
                double dp = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dp += do_row[d] * v_head[j * D + d];
                const double ds = p * (dp - delta[flat]) + (grad_in ? grad_in[flat * N + j] : 0.0);
                for (int64_t d = 0; d < D; ++d)
                    dq_row[d] += scale * ds * k_head[j * D + d];
                if (go) go[j] = ds;
            }
        }
        free(s);
    }
}

/*
 * dK and dV for the listed key rows; key row flat index (b*Hkv + g)*N + j.
 * Sums over every query head of the group and every query row i with
 * j in J_i.  lse, delta: full [B,Hq,N] arrays, read for the rows involved;
 * bias and grad_in as for orc_bwd_dq_rows (or NULL).
 *   dk, dv [nkrows, D].
 */
void orc_bwd_dkv_rows(const double *q, const double *k, const double *v, const double *dO,
                      const double *lse, const double *delta, const double *bias,
                      const double *grad_in,
                      int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t D,
                      double scale, int causal, int64_t window, const int64_t *krows,
                      int64_t nkrows, double *dk, double *dv)
{
    (void)B;
    const int64_t group = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nkrows; ++r) {
        const int64_t flat = krows ? krows[r] : r;
        const int64_t j = flat % N;
        const int64_t bg = flat / N;
        const int64_t b = bg / Hkv, g = bg % Hkv;
        const double *k_row = k + flat * D;
        const double *v_row = v + flat * D;
        double *dk_row = dk + r * D;
        double *dv_row = dv + r * D;
        for (int64_t d = 0; d < D; ++d) { dk_row[d] = 0.0; dv_row[d] = 0.0; }

        for (int64_t h = g * group; h < (g + 1) * group; ++h) {
            /* j in J_i  <=>  j <= i (causal) and i < j + W (window) */
            const int64_t i0 = causal ? j : 0;
            const int64_t i1 = (causal && window > 0 && j + window < N) ? j + window : N;
            for (int64_t i = i0; i < i1; ++i) {
                const int64_t qflat = (b * Hq + h) * N + i;
                const double *q_row = q + qflat * D;
                const double *do_row = dO + qflat * D;
                double dot = 0.0, dp = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    dot += q_row[d] * k_row[d];
                    dp += do_row[d] * v_row[d];
                }
                const double b_ij = bias ? bias[qflat * N + j] : 0.0;
                const double p = exp(scale * dot + b_ij - lse[qflat]);
                const double ds = p * (dp - delta[qflat]) + (grad_in ? grad_in[qflat * N + j] : 0.0);
                for (int64_t d = 0; d < D; ++d) {
                    dv_row[d] += p * do_row[d];
                    dk_row[d] += scale * ds * q_row[d];
                }
            }
        }
    }
}
