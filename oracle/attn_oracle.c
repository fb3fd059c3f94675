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
 * Dropout (oracle_attn_fwd_dropout / oracle_attn_bwd_dropout, at the end of this
 * file) multiplies each probability by a keep factor drawn from Philox4x32-10; the
 * definition is written out there.
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

/*
 * Dropout on the attention probabilities ("Understanding FlashAttention, Part 2",
 * section 2.4: the recomputing backward "also covers masking and dropout").  The
 * pages fix no random-number semantics; this library defines them:
 *
 *   Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
 *   as 1, 2, 3", SC 2011): counter (c0, c1, c2, c3), key (k0, k1); ten rounds of
 *     (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 *   with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by (0x9E3779B9, 0xBB67AE85)
 *   after every round.
 *
 *   Element (bh, i, j) (head bh, query i, key j) reads byte j mod 16 of
 *   Philox(counter = (j / 16, i, bh, 0), key = (seed_lo, seed_hi)), bytes taken
 *   little-endian from the four output words in order.  It is kept iff that byte is
 *   >= t, t = round(256 p) in 0..255 (so the drop probability is t / 256), and a kept
 *   probability is scaled by 1 / (1 - t / 256):
 *     O = (P o Z) V,   Z_ij = keep_ij * 256 / (256 - t),
 *   while the saved logsumexp is still that of the scores (dropout comes after the
 *   softmax).  Backward: dV = (P o Z)^T dO, dP~ = dO V^T, dS = P o (Z o dP~ - c) with
 *   c_i = sum_k P_ik Z_ik dP~_ik (= rowsum(dO o O)), dQ = scale dS K, dK = scale dS^T Q.
 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Z_ij of the definition above: 0 (dropped) or 256 / (256 - t) (kept). */
double oracle_dropout_factor(int64_t bh, int64_t i, int64_t j, int t, uint32_t seed_lo, uint32_t seed_hi)
{
    if (t <= 0) return 1.0;
    const uint32_t ctr[4] = {(uint32_t)(j / 16), (uint32_t)i, (uint32_t)bh, 0u};
    const uint32_t key[2] = {seed_lo, seed_hi};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    const int b = (int)(j % 16);
    const uint32_t byte = (w[b / 4] >> (8 * (b % 4))) & 0xFFu;
    return byte >= (uint32_t)t ? 256.0 / (256.0 - t) : 0.0;
}

/*
 * Forward with dropout: as oracle_attn_fwd (square or Nk >= N keys), with every
 * probability multiplied by its Z_ij before the sum over keys; lse is unchanged.
 * The arrays hold heads bh0 .. bh0 + BH - 1 (the head index enters the keep mask).
 */
int oracle_attn_fwd_dropout(const double *q, const double *k, const double *v,
                            int64_t BH, int64_t N, int64_t Nk, int64_t d, int causal, double scale,
                            int t, uint32_t seed_lo, uint32_t seed_hi, int64_t bh0,
                            const int64_t *rows, int64_t nrows, double *o, double *lse)
{
    if (BH < 0 || N < 1 || Nk < 1 || d < 1 || !q || !k || !v || !o || !lse) return -1;
    if (t < 0 || t > 255 || (causal && Nk < N)) return -1;
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
                for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    double pz = exp(s[j] - m) / l * oracle_dropout_factor(bh0 + bh, i, j, t, seed_lo, seed_hi);
                    const double *vj = vh + j * d;
                    for (int64_t c = 0; c < d; ++c) oi[c] += pz * vj[c];
                }
                lse[bh * nout + r] = m + log(l);
            }
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * Backward with dropout (definition above); arguments as oracle_attn_bwd plus t, the
 * seed and the first head's index bh0.  c_i is summed from its definition,
 * sum_k P_ik Z_ik dP~_ik.
 */
int oracle_attn_bwd_dropout(const double *q, const double *k, const double *v,
                            const double *dout, int64_t BH, int64_t N, int64_t Nk, int64_t d,
                            int causal, double scale, int t, uint32_t seed_lo, uint32_t seed_hi,
                            int64_t bh0,
                            const int64_t *qrows, int64_t nq,
                            const int64_t *kcols, int64_t nk,
                            double *dq, double *dk, double *dv)
{
    if (BH < 0 || N < 1 || Nk < 1 || d < 1 || !q || !k || !v || !dout) return -1;
    if (t < 0 || t > 255 || (causal && Nk < N)) return -1;
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

        /* 1. row statistics and c_i = sum_k P_ik Z_ik dP~_ik */
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
                    double z = oracle_dropout_factor(bh0 + bh, i, j, t, seed_lo, seed_hi);
                    double dpt = 0.0;                      /* dP~_ij = dO_i . V_j */
                    for (int64_t x = 0; x < d; ++x) dpt += doh[i * d + x] * vh[j * d + x];
                    acc += p * z * dpt;
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
                for (int64_t x = 0; x < d; ++x) g[x] = 0.0;
                for (int64_t j = 0; j < nkv; ++j) {
                    double sij = 0.0, dpt = 0.0;
                    for (int64_t x = 0; x < d; ++x) {
                        sij += qh[i * d + x] * kh[j * d + x];
                        dpt += doh[i * d + x] * vh[j * d + x];
                    }
                    double p = exp(scale * sij - m[i]) / l[i];
                    double z = oracle_dropout_factor(bh0 + bh, i, j, t, seed_lo, seed_hi);
                    double ds = p * (z * dpt - c[i]);
                    for (int64_t x = 0; x < d; ++x) g[x] += scale * ds * kh[j * d + x];
                }
            }
        }

        /* 3. dV_j = sum_i P_ij Z_ij dO_i ;  dK_j = scale * sum_i dS_ij Q_i */
        if (dk) {
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t r = 0; r < nko; ++r) {
                int64_t j = kcols ? kcols[r] : r;
                double *gk = dk + (bh * nko + r) * d;
                double *gv = dv + (bh * nko + r) * d;
                for (int64_t x = 0; x < d; ++x) { gk[x] = 0.0; gv[x] = 0.0; }
                int64_t i0 = causal ? j - (Nk - N) : 0;    /* queries that see key j */
                if (i0 < 0) i0 = 0;
                for (int64_t i = i0; i < N; ++i) {
                    double sij = 0.0, dpt = 0.0;
                    for (int64_t x = 0; x < d; ++x) {
                        sij += qh[i * d + x] * kh[j * d + x];
                        dpt += doh[i * d + x] * vh[j * d + x];
                    }
                    double p = exp(scale * sij - m[i]) / l[i];
                    double z = oracle_dropout_factor(bh0 + bh, i, j, t, seed_lo, seed_hi);
                    double ds = p * (z * dpt - c[i]);
                    for (int64_t x = 0; x < d; ++x) {
                        gv[x] += p * z * doh[i * d + x];
                        gk[x] += scale * ds * qh[i * d + x];
                    }
                }
            }
        }
    }
    free(m); free(l); free(c);
    return failed ? -1 : 0;
}
