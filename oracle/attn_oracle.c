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
 * Parity is pinned by the CPU tests (brute force, closed forms, invariants);
 * nothing here is "parity unpinned".
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
