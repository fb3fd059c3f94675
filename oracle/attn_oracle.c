/*
 * attn_oracle.c -- FP64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library) never calls it, and the two share no code.
 *
 * What it computes is the plain definition, written out entry by entry in
 * double precision, with no tiling, no online recurrence and no reordering:
 *
 *   S = scale * Q K^T                      ("FlashAttention hardware-aware
 *   P = softmax(S) row by row               analysis" (huaweicloud), section
 *   O = P V                                 one, part 2: the SDPA formula)
 *   LSE_i = m_i + ln l_i,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
 *                                          ("Understanding online softmax in
 *                                           Flash Attention from scratch",
 *                                           section 3.1: the m(x), l(x)
 *                                           decomposition)
 *
 * Causal masking keeps key j for query i iff j <= i; masked scores are -inf,
 * so their probabilities are exactly zero (huaweicloud page, section five,
 * part 3: the lower-triangular causal mask).  With Nq queries and Nk >= Nq
 * keys the triangle is aligned to the last key: query i sees keys
 * j <= i + (Nk - Nq), so the last query sees every key (a block of new
 * queries after Nk - Nq earlier positions); Nq = Nk is the square case.
 *
 * The backward pass is the chain rule of the same definition
 * ("Understanding FlashAttention, Part 2", section 2.4, Figs 16-19):
 *
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS_ij = P_ij * (dP_ij - c_i),   c_i = sum_k P_ik dP_ik   (softmax Jacobian)
 *   dQ = scale * dS K
 *   dK = scale * dS^T Q
 *
 * c_i is summed from its definition, not taken from rowsum(dO * O), so the
 * GPU path's shortcut through O is checked rather than shared.
 *
 * FP8 inputs with block scaling (huaweicloud page, section four, part 3: FP8
 * with per-block scale factors) are decoded to the real numbers they stand for
 * (oracle_dequant_e4m3) and then go through the same exact forward; the oracle
 * never rounds anything to FP8 itself.
 *
 * Layout: every tensor is [BH][N][d] row-major, d fastest, float64.
 * Threads: OpenMP over rows (and over key columns in the backward).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* s[j] = scale * <q_i, k_j> for the nkeys visible keys. */
static void score_row(const double *qi, const double *kh, int64_t nkeys,
                      int64_t d, double scale, double *s)
{
    for (int64_t j = 0; j < nkeys; ++j) {
        const double *kj = kh + j * d;
        double acc = 0.0;
        for (int64_t t = 0; t < d; ++t)
            acc += qi[t] * kj[t];
        s[j] = scale * acc;
    }
}

/* Row statistics of the softmax: m = max_j s_j, l = sum_j exp(s_j - m). */
static void row_stats(const double *s, int64_t nkeys, double *m_out, double *l_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j)
        l += exp(s[j] - m);
    *m_out = m;
    *l_out = l;
}

/* Keys visible to query i of Nq, with Nk keys (causal needs Nk >= Nq). */
static int64_t visible_keys(int64_t i, int64_t Nq, int64_t Nk, int causal)
{
    return causal ? (i + (Nk - Nq) + 1) : Nk;
}

/*
 * Forward.  q is [BH][N][d]; k and v are [BH][Nk][d] (Nk >= N when causal).
 * rows == NULL: every query row, o is [BH][N][d], lse is [BH][N].
 * rows != NULL: only rows[0..nrows), o is [BH][nrows][d], lse is [BH][nrows].
 * Returns 0, or -1 on a bad argument or an allocation failure.
 */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    int64_t BH, int64_t N, int64_t Nk, int64_t d, int causal, double scale,
                    const int64_t *rows, int64_t nrows, double *o, double *lse)
{
    if (BH < 0 || N < 1 || Nk < 1 || d < 1 || !q || !k || !v || !o || !lse) return -1;
    if (causal && Nk < N) return -1;
    int64_t nout = rows ? nrows : N;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= N) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4) collapse(2)
        for (int64_t bh = 0; bh < BH; ++bh) {
            for (int64_t r = 0; r < nout; ++r) {
                if (!s) continue;
                int64_t i = rows ? rows[r] : r;
                const double *qi = q + (bh * N + i) * d;
                const double *kh = k + bh * Nk * d;
                const double *vh = v + bh * Nk * d;
                int64_t nk = visible_keys(i, N, Nk, causal);
                double m, l;
                score_row(qi, kh, nk, d, scale, s);
                row_stats(s, nk, &m, &l);
                double *oi = o + (bh * nout + r) * d;
                for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    double p = exp(s[j] - m) / l;           /* P_ij */
                    const double *vj = vh + j * d;
                    for (int64_t t = 0; t < d; ++t) oi[t] += p * vj[t];
                }
                lse[bh * nout + r] = m + log(l);
            }
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * Backward.  Gradients of L = sum(dO * O) with respect to Q, K and V; q and dout
 * are [BH][N][d], k and v [BH][Nk][d] (Nk >= N when causal).
 * qrows == NULL: dq for every row ([BH][N][d]); else dq is [BH][nq][d] for
 * the listed query rows.  kcols == NULL: dk, dv for every key ([BH][Nk][d]);
 * else [BH][nk][d] for the listed keys.  Any of dq, dk/dv may be NULL to skip it.
 */
int oracle_attn_bwd(const double *q, const double *k, const double *v,
                    const double *dout, int64_t BH, int64_t N, int64_t Nk, int64_t d,
                    int causal, double scale,
                    const int64_t *qrows, int64_t nq,
                    const int64_t *kcols, int64_t nk,
                    double *dq, double *dk, double *dv)
{
    if (BH < 0 || N < 1 || Nk < 1 || d < 1 || !q || !k || !v || !dout) return -1;
    if (causal && Nk < N) return -1;
    if ((dk == NULL) != (dv == NULL)) return -1;
    int64_t nqo = qrows ? nq : N;
    int64_t nko = kcols ? nk : Nk;
    if (qrows)
        for (int64_t r = 0; r < nq; ++r)
            if (qrows[r] < 0 || qrows[r] >= N) return -1;
    if (kcols)
        for (int64_t r = 0; r < nk; ++r)
            if (kcols[r] < 0 || kcols[r] >= Nk) return -1;

    double *m = (double *)malloc(sizeof(double) * (size_t)N);
    double *l = (double *)malloc(sizeof(double) * (size_t)N);
    double *c = (double *)malloc(sizeof(double) * (size_t)N);
    if (!m || !l || !c) { free(m); free(l); free(c); return -1; }
    int failed = 0;

    for (int64_t bh = 0; bh < BH && !failed; ++bh) {
        const double *qh = q + bh * N * d;
        const double *kh = k + bh * Nk * d;
        const double *vh = v + bh * Nk * d;
        const double *doh = dout + bh * N * d;

        /* 1. per-row softmax statistics and c_i = sum_k P_ik dP_ik */
#pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
            if (!s) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 8)
            for (int64_t i = 0; i < N; ++i) {
                if (!s) continue;
                int64_t nkv = visible_keys(i, N, Nk, causal);
                score_row(qh + i * d, kh, nkv, d, scale, s);
                row_stats(s, nkv, &m[i], &l[i]);
                double acc = 0.0;
                for (int64_t j = 0; j < nkv; ++j) {
                    double p = exp(s[j] - m[i]) / l[i];
                    double dp = 0.0;                       /* dP_ij = dO_i . V_j */
                    for (int64_t t = 0; t < d; ++t) dp += doh[i * d + t] * vh[j * d + t];
                    acc += p * dp;
                }
                c[i] = acc;
            }
            free(s);
        }
        if (failed) break;

        /* 2. dQ_i = scale * sum_j dS_ij K_j */
        if (dq) {
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t r = 0; r < nqo; ++r) {
                int64_t i = qrows ? qrows[r] : r;
                int64_t nkv = visible_keys(i, N, Nk, causal);
                double *g = dq + (bh * nqo + r) * d;
                for (int64_t t = 0; t < d; ++t) g[t] = 0.0;
                for (int64_t j = 0; j < nkv; ++j) {
                    double sij = 0.0, dp = 0.0;
                    for (int64_t t = 0; t < d; ++t) {
                        sij += qh[i * d + t] * kh[j * d + t];
                        dp += doh[i * d + t] * vh[j * d + t];
                    }
                    double p = exp(scale * sij - m[i]) / l[i];
                    double ds = p * (dp - c[i]);
                    for (int64_t t = 0; t < d; ++t) g[t] += scale * ds * kh[j * d + t];
                }
            }
        }

        /* 3. dV_j = sum_i P_ij dO_i ;  dK_j = scale * sum_i dS_ij Q_i */
        if (dk) {
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t r = 0; r < nko; ++r) {
                int64_t j = kcols ? kcols[r] : r;
                double *gk = dk + (bh * nko + r) * d;
                double *gv = dv + (bh * nko + r) * d;
                for (int64_t t = 0; t < d; ++t) { gk[t] = 0.0; gv[t] = 0.0; }
                int64_t i0 = causal ? j - (Nk - N) : 0;    /* queries that see key j */
                if (i0 < 0) i0 = 0;
                for (int64_t i = i0; i < N; ++i) {
                    double sij = 0.0, dp = 0.0;
                    for (int64_t t = 0; t < d; ++t) {
                        sij += qh[i * d + t] * kh[j * d + t];
                        dp += doh[i * d + t] * vh[j * d + t];
                    }
                    double p = exp(scale * sij - m[i]) / l[i];
                    double ds = p * (dp - c[i]);
                    for (int64_t t = 0; t < d; ++t) {
                        gv[t] += p * doh[i * d + t];
                        gk[t] += scale * ds * qh[i * d + t];
                    }
                }
            }
        }
    }
    free(m); free(l); free(c);
    return failed ? -1 : 0;
}

/*
 * The value of one E4M3 code (the OCP 8-bit floating-point format, the variant
 * without infinities): bit 7 sign S, bits 6-3 exponent E (bias 7), bits 2-0
 * mantissa M.
 *   E = 0             (-1)^S * 2^-6 * (M / 8)          subnormals and +-0
 *   0 < E, not NaN    (-1)^S * 2^(E - 7) * (1 + M / 8)  largest: S.1111.110 = 448
 *   E = 15, M = 7     NaN
 */
double oracle_e4m3_value(uint8_t code)
{
    const int sgn = code >> 7;
    const int e = (code >> 3) & 15;
    const int man = code & 7;
    double mag;
    if (e == 15 && man == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)man / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)man / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/*
 * Block dequantisation: out[bh][n][c] = value(codes[bh][n][c]) * scales[bh][n / block_rows],
 * with codes [BH][N][d] E4M3 and scales [BH][ceil(N / block_rows)] float32 (one scale
 * per block of block_rows consecutive rows of one head).  Returns 0, or -1 on a bad
 * argument.
 */
int oracle_dequant_e4m3(const uint8_t *codes, const float *scales, int64_t BH, int64_t N,
                        int64_t d, int64_t block_rows, double *out)
{
    if (BH < 0 || N < 1 || d < 1 || block_rows < 1 || !codes || !scales || !out) return -1;
    const int64_t nblk = (N + block_rows - 1) / block_rows;
#pragma omp parallel for schedule(static)
    for (int64_t bh = 0; bh < BH; ++bh)
        for (int64_t n = 0; n < N; ++n) {
            const double sc = (double)scales[bh * nblk + n / block_rows];
            const int64_t base = (bh * N + n) * d;
            for (int64_t c = 0; c < d; ++c)
                out[base + c] = oracle_e4m3_value(codes[base + c]) * sc;
        }
    return 0;
}
