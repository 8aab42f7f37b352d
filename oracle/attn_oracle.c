/*
 * Attention-forward oracle: a plain, slow, fp64 CPU statement of what the
 * fused attention forward computes.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg load it; the product path
 * never does, and this file shares no code, header or constant with the CUDA
 * library.
 *
 * Sources (the three pages this project follows):
 *   - "flash-attn 实现 prefill 阶段" (dingfen.github.io), section 问题分析:
 *     tensors are [b, h, sq, d]; attn = softmax(Q K^T / sqrt(d)) V.
 *   - flash-attention-minimal flash.cu, forward_kernel: the scale is applied
 *     after the dot product (S = (Q.K) * softmax_scale), softmax uses the
 *     natural exponent, and the running statistics start at m = -inf, l = 0,
 *     O = 0 (host function forward()).
 *   - "05 · kernel 工程与四代演化", section 2.1: `causal` is one of the
 *     instantiation axes; the pages do not spell the mask out.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - causal mask, bottom-right aligned: key j is visible to query i iff
 *     j <= i + (sk - sq)  (plain j <= i when sq == sk);
 *   - a row that sees no key at all has O = 0 and LSE = -inf;
 *   - LSE is the natural log-sum-exp of the scaled logits: m + ln(l);
 *   - keys j >= sk do not exist (the minimal kernel's last tile reads past
 *     the end; here the loops simply stop at sk).
 *
 * Two computations are provided:
 *   oracle_attn_fwd_f64 / oracle_attn_head_rows_f64: the definition.  S is
 *     materialised one query row at a time (softmax is row-wise), then a
 *     two-pass softmax (max, then sum of exp) and the P.V product.
 *   oracle_attn_online_f64: the flash-attention-minimal recurrence (outer loop
 *     over K/V tiles of Bc keys, running m and l, O rescaled on every tile),
 *     restated in fp64 so that its algebra can be checked against the
 *     definition.
 * and, for the backward pass (end of the file): the gradients dQ, dK, dV of
 * the forward by definition (oracle_attn_bwd_f64), the same for selected
 * query rows or keys of one head (for spot checks of large problems), and
 * the probabilities P themselves (used to size error bounds); and the
 * KV-cache forward (oracle_attn_fwd_kvcache_f64): the cache write of new
 * tokens followed by the definition over each batch element's valid keys.
 * Parity is pinned by the CPU tests (brute force, closed forms, invariants,
 * finite differences of the forward for the gradients); nothing here is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_NOMEM -2

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Last key index visible to query row i (inclusive), or sk-1 without mask. */
static int64_t last_visible_key(int64_t i, int64_t sq, int64_t sk, int causal)
{
    int64_t last = sk - 1;
    if (causal) {
        int64_t diag = i + (sk - sq);
        if (diag < last) last = diag;
    }
    return last; /* may be < 0: the row sees no key */
}

/*
 * One query row of one head, straight from the definition.
 *   q: [d], K, V: [sk, d], srow: scratch of sk doubles, o: [d] out.
 */
static void row_by_definition(const double *q, const double *K, const double *V,
                              int64_t i, int64_t sq, int64_t sk, int64_t d,
                              int causal, double scale, double *srow,
                              double *o, double *lse)
{
    int64_t last = last_visible_key(i, sq, sk, causal);
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (last < 0) {
        *lse = -INFINITY;
        return;
    }
    int64_t n = last + 1; /* keys 0..last take part; the rest are masked out */

    /* S[i, j] = scale * sum_k Q[i, k] K[j, k] */
    for (int64_t j = 0; j < n; ++j) {
        const double *kj = K + j * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];
        srow[j] = dot * scale;
    }
    /* pass 1: row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (srow[j] > m) m = srow[j];
    /* pass 2: l = sum exp(S - m), P = exp(S - m) / l */
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        srow[j] = exp(srow[j] - m);
        l += srow[j];
    }
    for (int64_t j = 0; j < n; ++j) srow[j] /= l;
    /* O[i, :] = sum_j P[i, j] V[j, :] */
    for (int64_t j = 0; j < n; ++j) {
        const double *vj = V + j * d;
        double p = srow[j];
        for (int64_t c = 0; c < d; ++c) o[c] += p * vj[c];
    }
    *lse = m + log(l);
}

static int check_dims(int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d)
{
    if (b < 0 || h < 0 || sq < 0 || sk < 0 || d <= 0) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/*
 * Full forward by definition.  q, o: [b, h, sq, d]; k, v: [b, h, sk, d];
 * lse: [b, h, sq] (may be NULL).  All contiguous fp64.
 */
int oracle_attn_fwd_f64(const double *q, const double *k, const double *v,
                        double *o, double *lse, int64_t b, int64_t h,
                        int64_t sq, int64_t sk, int64_t d, int causal,
                        double scale)
{
    if (check_dims(b, h, sq, sk, d) != ORACLE_OK) return ORACLE_ERR_ARG;
    int64_t bh = b * h;
    int64_t total = bh * sq;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        if (!srow) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < total; ++r) {
                int64_t head = r / sq, i = r % sq;
                const double *Qh = q + head * sq * d;
                const double *Kh = k + head * sk * d;
                const double *Vh = v + head * sk * d;
                double l_out;
                row_by_definition(Qh + i * d, Kh, Vh, i, sq, sk, d, causal,
                                  scale, srow, o + r * d, &l_out);
                if (lse) lse[r] = l_out;
            }
            free(srow);
        }
    }
    return err;
}

/*
 * Selected rows of one head, by definition (for spot checks of large
 * problems).  q_head: [sq, d]; k_head, v_head: [sk, d]; rows: nrows query
 * indices; o_rows: [nrows, d]; lse_rows: [nrows].
 */
int oracle_attn_head_rows_f64(const double *q_head, const double *k_head,
                              const double *v_head, int64_t sq, int64_t sk,
                              int64_t d, int causal, double scale,
                              const int64_t *rows, int64_t nrows,
                              double *o_rows, double *lse_rows)
{
    if (check_dims(1, 1, sq, sk, d) != ORACLE_OK || nrows < 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= sq) return ORACLE_ERR_ARG;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        if (!srow) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < nrows; ++t) {
                int64_t i = rows[t];
                row_by_definition(q_head + i * d, k_head, v_head, i, sq, sk, d,
                                  causal, scale, srow, o_rows + t * d,
                                  &lse_rows[t]);
            }
            free(srow);
        }
    }
    return err;
}

/*
 * The flash-attention-minimal recurrence, restated in fp64 (forward_kernel):
 * for each K/V tile of Bc keys, for each query row:
 *   S = scale * Q_i K_j^T over the tile, row_m = max S, P = exp(S - row_m),
 *   row_l = sum P;  m_new = max(m_prev, row_m);
 *   l_new = exp(m_prev - m_new) l_prev + exp(row_m - m_new) row_l;
 *   O = (1/l_new) (l_prev exp(m_prev - m_new) O + exp(row_m - m_new) P V);
 * starting from m = -inf, l = 0, O = 0.  Masked or absent keys take no part;
 * a tile with no visible key for a row leaves that row unchanged.
 */
int oracle_attn_online_f64(const double *q, const double *k, const double *v,
                           double *o, double *lse, int64_t b, int64_t h,
                           int64_t sq, int64_t sk, int64_t d, int causal,
                           double scale, int64_t bc)
{
    if (check_dims(b, h, sq, sk, d) != ORACLE_OK || bc <= 0) return ORACLE_ERR_ARG;
    int64_t bh = b * h;
    int64_t total = bh * sq;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)bc);
        double *pv = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !pv) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < total; ++r) {
                int64_t head = r / sq, i = r % sq;
                const double *qi = q + head * sq * d + i * d;
                const double *Kh = k + head * sk * d;
                const double *Vh = v + head * sk * d;
                double *oi = o + r * d;
                double m_prev = -INFINITY, l_prev = 0.0;
                for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
                int64_t last = last_visible_key(i, sq, sk, causal);
                for (int64_t j0 = 0; j0 < sk; j0 += bc) {
                    int64_t j1 = j0 + bc < sk ? j0 + bc : sk;
                    if (j1 - 1 > last) j1 = last + 1; /* masked keys drop out */
                    int64_t n = j1 - j0;
                    if (n <= 0) continue;
                    double row_m = -INFINITY;
                    for (int64_t y = 0; y < n; ++y) {
                        const double *ky = Kh + (j0 + y) * d;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += qi[c] * ky[c];
                        s[y] = dot * scale;
                        if (s[y] > row_m) row_m = s[y];
                    }
                    double row_l = 0.0;
                    for (int64_t y = 0; y < n; ++y) {
                        s[y] = exp(s[y] - row_m);
                        row_l += s[y];
                    }
                    double m_new = m_prev > row_m ? m_prev : row_m;
                    double a_prev = exp(m_prev - m_new); /* 0 on the first tile */
                    double a_cur = exp(row_m - m_new);
                    double l_new = a_prev * l_prev + a_cur * row_l;
                    for (int64_t c = 0; c < d; ++c) {
                        double acc = 0.0;
                        for (int64_t y = 0; y < n; ++y) acc += s[y] * Vh[(j0 + y) * d + c];
                        pv[c] = acc;
                    }
                    for (int64_t c = 0; c < d; ++c)
                        oi[c] = (l_prev * a_prev * oi[c] + a_cur * pv[c]) / l_new;
                    m_prev = m_new;
                    l_prev = l_new;
                }
                if (lse) lse[r] = (l_prev > 0.0) ? m_prev + log(l_prev) : -INFINITY;
            }
        }
        free(s);
        free(pv);
    }
    return err;
}

/* ================================================================ backward
 *
 * Gradients of the forward above.  The pages name a backward pass (the
 * exported bwd / varlen_bwd entry points of "05 · kernel 工程与四代演化"
 * 6.1) but do not state it, so this is the chain rule through the
 * definition.  For a scalar loss L with dO = dL/dO given:
 *   O = P V                  ->  dV = P^T dO,   dP = dO V^T
 *   P[i, :] = softmax(S[i, :])
 *                            ->  dS[i, j] = P[i, j] (dP[i, j] - D[i]),
 *                                D[i] = sum_t P[i, t] dP[i, t]
 *   S = scale Q K^T          ->  dQ = scale dS K,   dK = scale dS^T Q
 * Masked keys have P = 0 and take no part; a row that sees no key has P = 0
 * throughout, so its dQ is 0 and it adds nothing to dK or dV.
 */

/* P[i, 0..sk) of one query row by definition (two-pass softmax); masked
 * keys get 0.  Returns the number of visible keys (0: the row is all 0). */
static int64_t probs_row_by_definition(const double *qi, const double *K, int64_t i,
                                       int64_t sq, int64_t sk, int64_t d, int causal,
                                       double scale, double *prow)
{
    int64_t last = last_visible_key(i, sq, sk, causal);
    for (int64_t j = 0; j < sk; ++j) prow[j] = 0.0;
    if (last < 0) return 0;
    int64_t n = 1 + last; /* visible keys 0..last */
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        const double *kj = K + j * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
        prow[j] = dot * scale;
        if (prow[j] > m) m = prow[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        prow[j] = exp(prow[j] - m);
        l += prow[j];
    }
    for (int64_t j = 0; j < n; ++j) prow[j] /= l;
    return n;
}

/* The probabilities P = softmax(scale Q K^T [+ causal]) themselves:
 * p [b, h, sq, sk] (used to size error bounds of the gradients). */
int oracle_attn_probs_f64(const double *q, const double *k, double *p, int64_t b,
                          int64_t h, int64_t sq, int64_t sk, int64_t d, int causal,
                          double scale)
{
    if (check_dims(b, h, sq, sk, d) != ORACLE_OK) return ORACLE_ERR_ARG;
    int64_t total = b * h * sq;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < total; ++r) {
        int64_t head = r / sq, i = r % sq;
        probs_row_by_definition(q + r * d, k + head * sk * d, i, sq, sk, d, causal, scale,
                                p + r * sk);
    }
    return ORACLE_OK;
}

/*
 * Full backward by definition.  q, dout, dq: [b, h, sq, d]; k, v, dk, dv:
 * [b, h, sk, d].  P and dP are materialised per head ([sq, sk] each).
 */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v,
                        const double *dout, double *dq, double *dk, double *dv,
                        int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d,
                        int causal, double scale)
{
    if (check_dims(b, h, sq, sk, d) != ORACLE_OK) return ORACLE_ERR_ARG;
    int64_t bh = b * h;
    for (int64_t x = 0; x < bh * sq * d; ++x) dq[x] = 0.0;
    for (int64_t x = 0; x < bh * sk * d; ++x) dk[x] = dv[x] = 0.0;
    if (sq == 0 || sk == 0) return ORACLE_OK;
    double *P = (double *)malloc(sizeof(double) * (size_t)(sq * sk));
    double *dP = (double *)malloc(sizeof(double) * (size_t)(sq * sk));
    if (!P || !dP) {
        free(P);
        free(dP);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t hd = 0; hd < bh; ++hd) {
        const double *Q = q + hd * sq * d, *K = k + hd * sk * d, *V = v + hd * sk * d;
        const double *dO = dout + hd * sq * d;
        double *dQ = dq + hd * sq * d, *dK = dk + hd * sk * d, *dV = dv + hd * sk * d;
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t i = 0; i < sq; ++i) {
            probs_row_by_definition(Q + i * d, K, i, sq, sk, d, causal, scale, P + i * sk);
            /* dP = dO V^T */
            for (int64_t j = 0; j < sk; ++j) {
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += dO[i * d + c] * V[j * d + c];
                dP[i * sk + j] = acc;
            }
            /* D[i] = sum_t P[i, t] dP[i, t];  dS (kept in dP) = P (dP - D) */
            double Di = 0.0;
            for (int64_t t = 0; t < sk; ++t) Di += P[i * sk + t] * dP[i * sk + t];
            for (int64_t j = 0; j < sk; ++j) dP[i * sk + j] = P[i * sk + j] * (dP[i * sk + j] - Di);
            /* dQ = scale dS K */
            for (int64_t c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int64_t j = 0; j < sk; ++j) acc += dP[i * sk + j] * K[j * d + c];
                dQ[i * d + c] = scale * acc;
            }
        }
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t j = 0; j < sk; ++j) {
            /* dV = P^T dO,  dK = scale dS^T Q */
            for (int64_t c = 0; c < d; ++c) {
                double av = 0.0, ak = 0.0;
                for (int64_t i = 0; i < sq; ++i) {
                    av += P[i * sk + j] * dO[i * d + c];
                    ak += dP[i * sk + j] * Q[i * d + c];
                }
                dV[j * d + c] = av;
                dK[j * d + c] = scale * ak;
            }
        }
    }
    free(P);
    free(dP);
    return ORACLE_OK;
}

/*
 * dQ for selected query rows of one head (for spot checks of large
 * problems): the same definition, one row at a time.  q_head, do_head:
 * [sq, d]; k_head, v_head: [sk, d]; dq_rows: [nrows, d].
 */
int oracle_attn_bwd_dq_rows_f64(const double *q_head, const double *k_head,
                                const double *v_head, const double *do_head,
                                int64_t sq, int64_t sk, int64_t d, int causal,
                                double scale, const int64_t *rows, int64_t nrows,
                                double *dq_rows)
{
    if (check_dims(1, 1, sq, sk, d) != ORACLE_OK || nrows < 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= sq) return ORACLE_ERR_ARG;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *prow = (double *)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        double *dprow = (double *)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        if (!prow || !dprow) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < nrows; ++t) {
                int64_t i = rows[t];
                const double *dOi = do_head + i * d;
                probs_row_by_definition(q_head + i * d, k_head, i, sq, sk, d, causal, scale, prow);
                double Di = 0.0;
                for (int64_t j = 0; j < sk; ++j) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; ++c) acc += dOi[c] * v_head[j * d + c];
                    dprow[j] = acc;
                    Di += prow[j] * acc;
                }
                for (int64_t c = 0; c < d; ++c) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < sk; ++j)
                        acc += prow[j] * (dprow[j] - Di) * k_head[j * d + c];
                    dq_rows[t * d + c] = scale * acc;
                }
            }
        }
        free(prow);
        free(dprow);
    }
    return err;
}

/*
 * dK and dV for selected keys of one head.  Every query row's softmax
 * (its max m[i] and sum l[i]) and D[i] are computed first, by definition;
 * then for each selected key j and each row i that sees it:
 *   P[i, j] = exp(S[i, j] - m[i]) / l[i],  dP[i, j] = dO[i] . V[j],
 *   dV[j] += P[i, j] dO[i],  dK[j] += scale P[i, j] (dP[i, j] - D[i]) Q[i].
 * dk_cols, dv_cols: [ncols, d].
 */
int oracle_attn_bwd_dkv_cols_f64(const double *q_head, const double *k_head,
                                 const double *v_head, const double *do_head,
                                 int64_t sq, int64_t sk, int64_t d, int causal,
                                 double scale, const int64_t *cols, int64_t ncols,
                                 double *dk_cols, double *dv_cols)
{
    if (check_dims(1, 1, sq, sk, d) != ORACLE_OK || ncols < 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < ncols; ++t)
        if (cols[t] < 0 || cols[t] >= sk) return ORACLE_ERR_ARG;
    double *m = (double *)malloc(sizeof(double) * (size_t)(sq > 0 ? sq : 1));
    double *l = (double *)malloc(sizeof(double) * (size_t)(sq > 0 ? sq : 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(sq > 0 ? sq : 1));
    if (!m || !l || !D) {
        free(m);
        free(l);
        free(D);
        return ORACLE_ERR_NOMEM;
    }
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        if (!srow) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < sq; ++i) {
                const double *qi = q_head + i * d, *dOi = do_head + i * d;
                int64_t n = last_visible_key(i, sq, sk, causal) + 1;
                double mi = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += qi[c] * k_head[j * d + c];
                    srow[j] = scale * dot;
                    if (srow[j] > mi) mi = srow[j];
                }
                double li = 0.0, Di = 0.0;
                for (int64_t j = 0; j < n; ++j) li += exp(srow[j] - mi);
                for (int64_t j = 0; j < n; ++j) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; ++c) acc += dOi[c] * v_head[j * d + c];
                    Di += exp(srow[j] - mi) / li * acc;
                }
                m[i] = mi;
                l[i] = li;
                D[i] = Di;
            }
        }
        free(srow);
    }
    if (err != ORACLE_OK) {
        free(m);
        free(l);
        free(D);
        return err;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < ncols; ++t) {
        int64_t j = cols[t];
        const double *kj = k_head + j * d, *vj = v_head + j * d;
        double *dKj = dk_cols + t * d, *dVj = dv_cols + t * d;
        for (int64_t c = 0; c < d; ++c) dKj[c] = dVj[c] = 0.0;
        for (int64_t i = 0; i < sq; ++i) {
            if (j > last_visible_key(i, sq, sk, causal)) continue;
            const double *qi = q_head + i * d, *dOi = do_head + i * d;
            double s = 0.0, dp = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                s += qi[c] * kj[c];
                dp += dOi[c] * vj[c];
            }
            double p = exp(s * scale - m[i]) / l[i];
            double ds = p * (dp - D[i]);
            for (int64_t c = 0; c < d; ++c) {
                dVj[c] += p * dOi[c];
                dKj[c] += scale * ds * qi[c];
            }
        }
    }
    free(m);
    free(l);
    free(D);
    return ORACLE_OK;
}

/*
 * KV-cache forward.  "05 · kernel 工程与四代演化", section 6.1, names a
 * fwd_kvcache entry point without defining it; the reading taken here:
 *   1. for each batch element e, with L0 = cache_len[e] clamped to
 *      [0, s_cache], row t of the new keys and values goes to position
 *      L0 + t of the cache; rows that would fall at or past s_cache are
 *      dropped;
 *   2. every query row of e attends, by definition, to the first
 *      L = min(L0 + s_new, s_cache) keys of e's cache (causal mask
 *      bottom-right aligned to L, as for the plain forward with sk = L).
 * k_cache, v_cache: [b, h, s_cache, d], updated in place; k_new, v_new:
 * [b, h, s_new, d] (may be NULL when s_new == 0); cache_len: [b];
 * q, o: [b, h, sq, d]; lse: [b, h, sq] (may be NULL).
 */
static int64_t clamp_len(int64_t len, int64_t cap)
{
    if (len < 0) return 0;
    return len > cap ? cap : len;
}

int oracle_attn_fwd_kvcache_f64(const double *q, double *k_cache, double *v_cache,
                                const double *k_new, const double *v_new,
                                const int64_t *cache_len, double *o, double *lse,
                                int64_t b, int64_t h, int64_t sq, int64_t s_cache,
                                int64_t s_new, int64_t d, int causal, double scale)
{
    if (check_dims(b, h, sq, s_cache, d) != ORACLE_OK || s_new < 0) return ORACLE_ERR_ARG;
    if (s_new > 0 && (!k_new || !v_new)) return ORACLE_ERR_ARG;
    /* step 1: the new rows go into the cache after the valid ones */
    for (int64_t e = 0; e < b; ++e) {
        int64_t start = clamp_len(cache_len[e], s_cache);
        for (int64_t head = 0; head < h; ++head) {
            int64_t plane = e * h + head;
            for (int64_t t = 0; t < s_new; ++t) {
                int64_t pos = start + t;
                if (pos >= s_cache) break; /* no room left in the cache */
                memcpy(k_cache + (plane * s_cache + pos) * d, k_new + (plane * s_new + t) * d,
                       sizeof(double) * (size_t)d);
                memcpy(v_cache + (plane * s_cache + pos) * d, v_new + (plane * s_new + t) * d,
                       sizeof(double) * (size_t)d);
            }
        }
    }
    /* step 2: attention over the valid prefix of each element's cache */
    int64_t total = b * h * sq;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(s_cache > 0 ? s_cache : 1));
        if (!srow) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < total; ++r) {
                int64_t plane = r / sq, i = r % sq;
                int64_t e = plane / h;
                int64_t valid = clamp_len(cache_len[e], s_cache) + s_new;
                if (valid > s_cache) valid = s_cache;
                double l_out;
                row_by_definition(q + r * d, k_cache + plane * s_cache * d, v_cache + plane * s_cache * d,
                                  i, sq, valid, d, causal, scale, srow, o + r * d, &l_out);
                if (lse) lse[r] = l_out;
            }
            free(srow);
        }
    }
    return err;
}
