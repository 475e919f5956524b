/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU implementation of exact softmax attention, written
 * from the definition the pages give, used to check the CUDA path.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it;
 * the library's compute path never calls it and shares no code with it.
 *
 * What it computes (standard attention, "S = QK^T/sqrt(d) -> P = softmax(S)
 * -> O = PV", clxhxhhr.top S23-J17 §3; also ans20xx.com day14, "online
 * softmax 的最小直觉"):
 *
 *   for batch b, query head h, query row i, with KV head g = h / (Hq/Hkv)
 *   (contiguous groups: "每 4 个 Q 头共享 1 个 KV 头", lei6393.com §2.3)
 *   and allowed key set J_i:
 *       s_ij  = scale * sum_c q[b,i,h,c] * k[b,j,g,c]
 *       m_i   = max_{j in J_i} s_ij
 *       P_ij  = exp(s_ij - m_i) / sum_{j in J_i} exp(s_ij - m_i)
 *       O[i]  = sum_{j in J_i} P_ij v[b,j,g,:]
 *       lse_i = m_i + ln sum_{j in J_i} exp(s_ij - m_i)
 *
 *   J_i holds the keys j < Lk that the key_padding_mask keeps (True = keep,
 *   lei6393.com §2.5) and, when causal, j <= i + (Lk - Lq) (causal includes
 *   the diagonal and is aligned bottom-right when Lq != Lk; the pages are
 *   silent on that case).  A row with an empty J_i, or a query row that the
 *   padding mask drops, gets O = 0 and lse = -inf.
 *
 * Every score row is materialised in full (S_i, then P_i) before O_i is
 * formed; nothing is blocked or fused.  Subtracting m_i inside the exponent
 * leaves the value of the definition unchanged.
 *
 * A second routine, used only to check that the tiled method reaches the same
 * result, runs the online-softmax recurrence over key blocks of size beta in
 * one of the two forms the pages print:
 *   form 0 (clxhxhhr.top S23-J17 §3.1): running max m, exp-sum l relative to m,
 *          value sum u with the same weights; on a max change
 *          r = exp(m_old - m_new) rescales l and u; O = u / l at the end.
 *   form 1 (ans20xx.com day14 online-softmax pseudocode): m, l and a
 *          normalised output o, updated as
 *          o = (alpha*l*o + p.V) / l_new with alpha = exp(m - m_new).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int check_dims(int B, int Hq, int Hkv, int Lq, int Lk, int d)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0 || d <= 0)
        return ORACLE_EINVAL;
    if (Hq % Hkv != 0)
        return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* Is key j visible to query row i of batch b? */
static int key_allowed(int i, int j, int Lq, int Lk, int causal,
                       const unsigned char *kmask_b)
{
    if (kmask_b && !kmask_b[j])
        return 0;
    if (causal && j > i + (Lk - Lq))
        return 0;
    return 1;
}

/* Index helpers: q and o are (B, Lq, Hq, d); k and v are (B, Lk, Hkv, d). */
static inline size_t qidx(int b, int i, int h, int c, int Lq, int Hq, int d)
{
    return (((size_t)b * Lq + i) * Hq + h) * d + c;
}
static inline size_t kidx(int b, int j, int g, int c, int Lk, int Hkv, int d)
{
    return (((size_t)b * Lk + j) * Hkv + g) * d + c;
}

/*
 * One query row by the definition.  s and p are caller-provided scratch rows
 * of length Lk.  If p_row is not NULL the probabilities are copied there.
 */
static void attention_row(const double *q, const double *k, const double *v,
                          const unsigned char *kpm, int B, int Hq, int Hkv,
                          int Lq, int Lk, int d, int causal, double scale,
                          int b, int h, int i, double *s, double *p,
                          double *o_row, double *lse_out, double *p_row)
{
    (void)B;
    const int group = Hq / Hkv;
    const int g = h / group;
    const unsigned char *kmask_b = kpm ? kpm + (size_t)b * Lk : NULL;
    int c, j, n_allowed = 0;
    double m = -INFINITY, denom = 0.0;

    /* query rows that the padding mask drops produce nothing */
    int row_is_token = 1;
    if (kpm && Lq == Lk && !kmask_b[i])
        row_is_token = 0;

    /* S_i: the full score row */
    for (j = 0; j < Lk; ++j) {
        if (!row_is_token || !key_allowed(i, j, Lq, Lk, causal, kmask_b)) {
            s[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (c = 0; c < d; ++c) {
            acc += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, g, c, Lk, Hkv, d)];
        }
        s[j] = scale * acc;
        n_allowed++;
        if (s[j] > m)
            m = s[j];
    }

    if (n_allowed == 0) {
        for (c = 0; c < d; ++c)
            o_row[c] = 0.0;
        *lse_out = -INFINITY;
        if (p_row)
            for (j = 0; j < Lk; ++j)
                p_row[j] = 0.0;
        return;
    }

    /* P_i = softmax(S_i) over the allowed keys */
    for (j = 0; j < Lk; ++j) {
        if (s[j] == -INFINITY) {
            p[j] = 0.0;
            continue;
        }
        p[j] = exp(s[j] - m);
        denom += p[j];
    }
    for (j = 0; j < Lk; ++j)
        p[j] /= denom;

    /* O_i = P_i V */
    for (c = 0; c < d; ++c) {
        double acc = 0.0;
        for (j = 0; j < Lk; ++j)
            acc += p[j] * v[kidx(b, j, g, c, Lk, Hkv, d)];
        o_row[c] = acc;
    }
    *lse_out = m + log(denom);
    if (p_row)
        memcpy(p_row, p, sizeof(double) * (size_t)Lk);
}

/*
 * Full attention.  q (B,Lq,Hq,d), k/v (B,Lk,Hkv,d), o (B,Lq,Hq,d),
 * lse (B,Hq,Lq).  key_padding_mask: NULL or (B,Lk) bytes, nonzero = keep.
 * probs: NULL or (B,Hq,Lq,Lk), receives every materialised P row.
 */
int oracle_attention(const double *q, const double *k, const double *v,
                     const unsigned char *key_padding_mask, double *o,
                     double *lse, double *probs, int B, int Hq, int Hkv,
                     int Lq, int Lk, int d, int causal, double scale)
{
    int rc = check_dims(B, Hq, Hkv, Lq, Lk, d);
    if (rc)
        return rc;
    if (key_padding_mask && Lq != Lk)
        return ORACLE_EINVAL;
    const long nrows = (long)B * Hq * Lq;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double *orow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !p || !orow) {
#pragma omp atomic write
            failed = 1;
        } else {
            long r;
#pragma omp for schedule(dynamic, 16)
            for (r = 0; r < nrows; ++r) {
                int b = (int)(r / ((long)Hq * Lq));
                int h = (int)((r / Lq) % Hq);
                int i = (int)(r % Lq);
                double l;
                double *prow = probs ? probs + (((size_t)b * Hq + h) * Lq + i) * (size_t)Lk : NULL;
                attention_row(q, k, v, key_padding_mask, B, Hq, Hkv, Lq, Lk, d,
                              causal, scale, b, h, i, s, p, orow, &l, prow);
                memcpy(o + qidx(b, i, h, 0, Lq, Hq, d), orow, sizeof(double) * (size_t)d);
                lse[((size_t)b * Hq + h) * Lq + i] = l;
            }
        }
        free(s);
        free(p);
        free(orow);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * Selected rows only.  rows holds nrows triples (b, h, i); o_rows is
 * (nrows, d) and lse_rows (nrows).  Used to check outputs of problems too
 * large to evaluate in full on the CPU.
 */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          const unsigned char *key_padding_mask,
                          const int *rows, int nrows, double *o_rows,
                          double *lse_rows, int B, int Hq, int Hkv, int Lq,
                          int Lk, int d, int causal, double scale)
{
    int rc = check_dims(B, Hq, Hkv, Lq, Lk, d);
    if (rc)
        return rc;
    if (key_padding_mask && Lq != Lk)
        return ORACLE_EINVAL;
    for (int r = 0; r < nrows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Lq)
            return ORACLE_EINVAL;
    }
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        if (!s || !p) {
#pragma omp atomic write
            failed = 1;
        } else {
            int r;
#pragma omp for schedule(dynamic, 4)
            for (r = 0; r < nrows; ++r) {
                attention_row(q, k, v, key_padding_mask, B, Hq, Hkv, Lq, Lk, d,
                              causal, scale, rows[3 * r], rows[3 * r + 1],
                              rows[3 * r + 2], s, p, o_rows + (size_t)r * d,
                              lse_rows + r, NULL);
            }
        }
        free(s);
        free(p);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * The online-softmax recurrence for selected rows, over key blocks of beta
 * consecutive key indices (the last block may be shorter).  form 0 is the
 * (m, l, u, r) recurrence, form 1 the normalised-o recurrence; see the file
 * header.  If trace is not NULL it receives, for the FIRST row only and after
 * every block, the triple (m, l, u[0]) (form 1 stores o[0] in place of u[0]);
 * it must hold 3 * ceil(Lk / beta) doubles.
 */
int oracle_online_rows(const double *q, const double *k, const double *v,
                       const unsigned char *key_padding_mask, const int *rows,
                       int nrows, double *o_rows, double *lse_rows, int B,
                       int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                       double scale, int beta, int form, double *trace)
{
    int rc = check_dims(B, Hq, Hkv, Lq, Lk, d);
    if (rc)
        return rc;
    if (beta <= 0 || (form != 0 && form != 1))
        return ORACLE_EINVAL;
    if (key_padding_mask && Lq != Lk)
        return ORACLE_EINVAL;
    double *s = (double *)malloc(sizeof(double) * (size_t)(beta));
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    double *pv = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !acc || !pv) {
        free(s);
        free(acc);
        free(pv);
        return ORACLE_ENOMEM;
    }
    const int group = Hq / Hkv;
    for (int r = 0; r < nrows; ++r) {
        const int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Lq) {
            free(s);
            free(acc);
            free(pv);
            return ORACLE_EINVAL;
        }
        const int g = h / group;
        const unsigned char *kmask_b = key_padding_mask ? key_padding_mask + (size_t)b * Lk : NULL;
        const int row_is_token = !(key_padding_mask && !kmask_b[i]);
        double m = -INFINITY, l = 0.0;
        for (int c = 0; c < d; ++c)
            acc[c] = 0.0;
        int blk = 0;
        for (int j0 = 0; j0 < Lk; j0 += beta, ++blk) {
            const int n = (Lk - j0 < beta) ? (Lk - j0) : beta;
            double m_blk = -INFINITY;
            for (int t = 0; t < n; ++t) {
                const int j = j0 + t;
                if (!row_is_token || !key_allowed(i, j, Lq, Lk, causal, kmask_b)) {
                    s[t] = -INFINITY;
                    continue;
                }
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, g, c, Lk, Hkv, d)];
                s[t] = scale * dot;
                if (s[t] > m_blk)
                    m_blk = s[t];
            }
            const double m_new = (m_blk > m) ? m_blk : m;
            if (m_new != -INFINITY) {
                /* r (form 0) and alpha (form 1) are the same factor */
                const double r_fac = (m == -INFINITY) ? 0.0 : exp(m - m_new);
                double psum = 0.0;
                for (int c = 0; c < d; ++c)
                    pv[c] = 0.0;
                for (int t = 0; t < n; ++t) {
                    if (s[t] == -INFINITY)
                        continue;
                    const double pt = exp(s[t] - m_new);
                    psum += pt;
                    for (int c = 0; c < d; ++c)
                        pv[c] += pt * v[kidx(b, j0 + t, g, c, Lk, Hkv, d)];
                }
                const double l_new = r_fac * l + psum;
                if (form == 0) {
                    for (int c = 0; c < d; ++c)
                        acc[c] = r_fac * acc[c] + pv[c];
                } else {
                    for (int c = 0; c < d; ++c)
                        acc[c] = (r_fac * l * acc[c] + pv[c]) / l_new;
                }
                m = m_new;
                l = l_new;
            }
            if (trace && r == 0) {
                trace[3 * blk + 0] = m;
                trace[3 * blk + 1] = l;
                trace[3 * blk + 2] = acc[0];
            }
        }
        double *o_row = o_rows + (size_t)r * d;
        if (l == 0.0) {
            for (int c = 0; c < d; ++c)
                o_row[c] = 0.0;
            lse_rows[r] = -INFINITY;
        } else {
            for (int c = 0; c < d; ++c)
                o_row[c] = (form == 0) ? acc[c] / l : acc[c];
            lse_rows[r] = m + log(l);
        }
    }
    free(s);
    free(acc);
    free(pv);
    return ORACLE_OK;
}

/*
 * Backward pass of the same attention (lei6393.com training-integration page,
 * §5.3: the backward recomputes the attention weights instead of storing the
 * O(N^2) matrix).  The pages give no formulas; these are the gradients of the
 * scalar sum(dout * O) with respect to q, k and v, from the chain rule through
 * the definition at the top of this file:
 *
 *   dP_ij = dout_i . v_j                               (O_i = sum_j P_ij v_j)
 *   dS_ij = P_ij * (dP_ij - sum_{k in J_i} P_ik dP_ik)  (Jacobian of the row softmax)
 *   dq_i  = scale * sum_j dS_ij k_j                    (s_ij = scale * q_i . k_j)
 *   dk_j  = scale * sum_{h in group, i} dS_ij q_i
 *   dv_j  = sum_{h in group, i} P_ij dout_i
 *
 * Each P row is materialised by the forward routine, then its dP and dS rows.
 * One (batch, KV head) pair per OpenMP task, so dk and dv are summed by one
 * thread.  dout is (B,Lq,Hq,d) like q; dq like q, dk and dv like k.
 */
int oracle_attention_backward(const double *q, const double *k, const double *v,
                              const double *dout,
                              const unsigned char *key_padding_mask,
                              double *dq, double *dk, double *dv, int B, int Hq,
                              int Hkv, int Lq, int Lk, int d, int causal,
                              double scale)
{
    int rc = check_dims(B, Hq, Hkv, Lq, Lk, d);
    if (rc)
        return rc;
    if (key_padding_mask && Lq != Lk)
        return ORACLE_EINVAL;
    const int group = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)B * Lq * Hq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Lk * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Lk * Hkv * d);
    const long npairs = (long)B * Hkv;
    int failed = 0;
#pragma omp parallel
    {
        const size_t nk = (size_t)(Lk > 0 ? Lk : 1);
        double *s = (double *)malloc(sizeof(double) * nk);
        double *p = (double *)malloc(sizeof(double) * nk);
        double *prow = (double *)malloc(sizeof(double) * nk);
        double *dp = (double *)malloc(sizeof(double) * nk);
        double *orow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !p || !prow || !dp || !orow) {
#pragma omp atomic write
            failed = 1;
        } else {
            long r;
#pragma omp for schedule(dynamic, 1)
            for (r = 0; r < npairs; ++r) {
                const int b = (int)(r / Hkv), g = (int)(r % Hkv);
                for (int h = g * group; h < (g + 1) * group; ++h) {
                    for (int i = 0; i < Lq; ++i) {
                        double lse;
                        attention_row(q, k, v, key_padding_mask, B, Hq, Hkv, Lq, Lk, d,
                                      causal, scale, b, h, i, s, p, orow, &lse, prow);
                        /* dP row and the softmax-weighted mean of dP */
                        double mean_dp = 0.0;
                        for (int j = 0; j < Lk; ++j) {
                            dp[j] = 0.0;
                            if (prow[j] == 0.0)
                                continue;
                            double acc = 0.0;
                            for (int c = 0; c < d; ++c)
                                acc += dout[qidx(b, i, h, c, Lq, Hq, d)] * v[kidx(b, j, g, c, Lk, Hkv, d)];
                            dp[j] = acc;
                            mean_dp += prow[j] * acc;
                        }
                        for (int j = 0; j < Lk; ++j) {
                            if (prow[j] == 0.0)
                                continue;
                            const double ds = prow[j] * (dp[j] - mean_dp);
                            for (int c = 0; c < d; ++c) {
                                dq[qidx(b, i, h, c, Lq, Hq, d)] += scale * ds * k[kidx(b, j, g, c, Lk, Hkv, d)];
                                dk[kidx(b, j, g, c, Lk, Hkv, d)] += scale * ds * q[qidx(b, i, h, c, Lq, Hq, d)];
                                dv[kidx(b, j, g, c, Lk, Hkv, d)] += prow[j] * dout[qidx(b, i, h, c, Lq, Hq, d)];
                            }
                        }
                    }
                }
            }
        }
        free(s);
        free(p);
        free(prow);
        free(dp);
        free(orow);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}
