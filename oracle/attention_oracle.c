/*
 * Oracle for exact (softmax) attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 CPU restatement of what the fused
 * attention forward computes.  Only tests/, the smoke check and the CPU
 * baseline leg of the benchmark may load this library; the product path
 * never does.  It shares no code, header or constant with the CUDA path.
 *
 * Definition followed (no tiling, no online rescaling, no fusion):
 *   "Parsing FlashAttention (2): FlashAttention-v1 forward pass", §1.1
 *   (S = Q K^T, P = softmax(S), O = P V) and §2.1 eqs (1)-(5) (safe softmax);
 *   "Online Softmax and FlashAttention" (course unit 12), causal-mask passage
 *   (M_ij = -inf for j > i, future weights exactly 0).
 * Readings of points the pages leave open:
 *   - the scale multiplies the fp64 dot product (it is not folded into Q);
 *   - LSE_i = m_i + ln(l_i) of the scaled, masked scores (natural log);
 *   - causal masking: query i of Nq sits at position Nk - Nq + i of the Nk
 *     keys and sees keys 0..Nk-Nq+i (square attention: keys 0..i).
 *
 * Inputs are 16-bit bit patterns (uint16) of bf16 or, for the fp16 variant
 * ("pwwt.cn FlashAttention/Triton walkthrough" §3.4 runs in fp16; §5 lists
 * fp16 among the extensions), IEEE binary16; each is widened to fp64
 * exactly.  Every floating-point step below runs in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Exact widening of an IEEE 754 binary16 bit pattern: sign bit, 5-bit
 * exponent with bias 15, 10-bit fraction; exponent 0 holds zeros and
 * subnormals (fraction * 2^-24), exponent 31 infinities and NaNs.
 */
double oracle_f16_to_double(uint16_t bits)
{
    int sign = bits >> 15;
    int e = (bits >> 10) & 31;
    int frac = bits & 1023;
    double mag;
    if (e == 0)
        mag = ldexp((double)frac, -24);
    else if (e == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), e - 25);
    return sign ? -mag : mag;
}

/* Element formats of the 16-bit inputs. */
enum { ORACLE_BF16 = 0, ORACLE_F16 = 1 };

static double widen(uint16_t bits, int fmt)
{
    return fmt == ORACLE_F16 ? oracle_f16_to_double(bits) : oracle_bf16_to_double(bits);
}

/*
 * One row of scores (page 1 §1.1; page 2 causal passage), inputs of format
 * fmt:
 *   s_j = scale * sum_t q_t * k_{j,t}     for visible j,
 *   s_j = -inf                           for j > i when causal.
 */
static void score_row_fmt(const uint16_t *q_row, const uint16_t *k, int64_t i,
                          int64_t n_keys, int64_t d, double scale, int causal,
                          int fmt, double *s)
{
    for (int64_t j = 0; j < n_keys; ++j) {
        if (causal && j > i) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t)
            dot += widen(q_row[t], fmt) * widen(k[j * d + t], fmt);
        s[j] = scale * dot;
    }
}

/*
 * Safe softmax of one vector (page 1 §2.1, eqs (1)-(5)):
 *   m = max_j x_j,  shifted_j = x_j - m,  f_j = exp(shifted_j),
 *   l = sum_j f_j,  p_j = f_j / l.
 * Entries equal to -inf give f_j = exp(-inf) = 0 exactly.  Any output
 * pointer may be NULL.  Requires at least one finite entry.
 */
void oracle_safe_softmax(const double *x, int64_t n, double *shifted,
                         double *p, double *m_out, double *l_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m) m = x[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double sh = x[j] - m;
        if (shifted) shifted[j] = sh;
        l += exp(sh);
    }
    if (p)
        for (int64_t j = 0; j < n; ++j) p[j] = exp(x[j] - m) / l;
    if (m_out) *m_out = m;
    if (l_out) *l_out = l;
}

/*
 * Full score block for rows [0, nq) of q against all nk keys; row r of q is
 * query index row_offset + r (used only by the causal test j > i).
 * s_out: nq x nk, row-major.
 */
void oracle_scores(const uint16_t *q, const uint16_t *k, int64_t nq,
                   int64_t nk, int64_t d, double scale, int causal,
                   int64_t row_offset, double *s_out)
{
    for (int64_t r = 0; r < nq; ++r)
        score_row_fmt(q + r * d, k, row_offset + r, nk, d, scale, causal,
                      ORACLE_BF16, s_out + r * nk);
}

/*
 * Attention forward for selected query rows of every (batch, head) slice,
 * with Nq queries against Nk keys.  Causal masking is aligned to the end of
 * the key sequence: query i sits at position Nk - Nq + i and sees keys
 * j <= Nk - Nq + i (for Nq == Nk this is the square rule j <= i).
 *   q       : [BH][Nq][d] 16-bit patterns of format fmt (ORACLE_BF16 / ORACLE_F16)
 *   k, v    : [BH][Nk][d] 16-bit patterns of format fmt
 *   rows    : n_rows query indices (each in [0, Nq)), applied to every slice;
 *             NULL means all rows (n_rows must then equal Nq)
 *   o_out   : [BH][n_rows][d] fp64,   O_i = sum_j P_ij v_j
 *   lse_out : [BH][n_rows]   fp64,   LSE_i = m_i + ln(l_i)
 *   p_out   : optional [BH][n_rows][Nk] fp64 probabilities (may be NULL)
 * Returns 0, or -1 on bad arguments / -2 on allocation failure.
 */
int oracle_attention_rect_fmt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int causal,
                              double scale, const int64_t *rows, int64_t n_rows,
                              double *o_out, double *lse_out, double *p_out, int n_threads,
                              int fmt)
{
    if (!q || !k || !v || !o_out || !lse_out) return -1;
    if (fmt != ORACLE_BF16 && fmt != ORACLE_F16) return -1;
    if (BH <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || n_rows <= 0) return -1;
    if (causal && Nq > Nk) return -1; /* some query would see no key */
    if (!rows && n_rows != Nq) return -1;
    for (int64_t r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= Nq) return -1;

    int failed = 0;
    int64_t tasks = BH * n_rows;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        double *p = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s || !p) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t task = 0; task < tasks; ++task) {
            if (!s || !p) continue;
            int64_t bh = task / n_rows;
            int64_t r = task % n_rows;
            int64_t i = rows ? rows[r] : r;
            const uint16_t *qh = q + (bh * Nq + i) * d;
            const uint16_t *kh = k + bh * Nk * d;
            const uint16_t *vh = v + bh * Nk * d;

            /* position of query i among the keys (end-aligned) */
            score_row_fmt(qh, kh, Nk - Nq + i, Nk, d, scale, causal, fmt, s);
            double m, l;
            oracle_safe_softmax(s, Nk, NULL, p, &m, &l);

            double *o = o_out + (bh * n_rows + r) * d;
            for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
            for (int64_t j = 0; j < Nk; ++j) {
                if (p[j] == 0.0) continue; /* masked keys add 0 * v_j */
                for (int64_t t = 0; t < d; ++t)
                    o[t] += p[j] * widen(vh[j * d + t], fmt);
            }
            lse_out[bh * n_rows + r] = m + log(l);
            if (p_out)
                memcpy(p_out + (bh * n_rows + r) * Nk, p,
                       (size_t)Nk * sizeof(double));
        }
        free(s);
        free(p);
    }
    return failed ? -2 : 0;
}

/*
 * Gradients of the attention forward (the backward pass by recomputation
 * that "Parsing FlashAttention (2)" §1 and "Online Softmax and
 * FlashAttention" name as the reason to keep the row statistics), written
 * from the definition rather than any tiling: for every query row i, with
 * s_ij the scaled, masked scores and P_ij = softmax_j(s_ij),
 *   dV_j  += P_ij dO_i                       (O = P V)
 *   dP_ij  = dO_i . V_j
 *   dS_ij  = P_ij (dP_ij - sum_k P_ik dP_ik)  (Jacobian of a softmax row)
 *   dQ_i   = scale * sum_j dS_ij K_j          (s = scale * Q K^T)
 *   dK_j  += scale * dS_ij Q_i.
 *   q, k, v, dout : [BH][N][d] 16-bit patterns of format fmt
 *   dq, dk, dv    : [BH][N][d] fp64, written
 * Square attention (causal: query i sees keys 0..i).  One (batch, head)
 * slice per OpenMP task.  Returns 0, -1 on bad arguments, -2 on allocation
 * failure.
 */
int oracle_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int64_t BH, int64_t N, int64_t d, int causal,
                         double scale, double *dq, double *dk, double *dv, int n_threads,
                         int fmt)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if (BH <= 0 || N <= 0 || d <= 0) return -1;
    if (fmt != ORACLE_BF16 && fmt != ORACLE_F16) return -1;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t bh = 0; bh < BH; ++bh) {
        const uint16_t *qh = q + bh * N * d, *kh = k + bh * N * d;
        const uint16_t *vh = v + bh * N * d, *doh = dout + bh * N * d;
        double *dqh = dq + bh * N * d, *dkh = dk + bh * N * d, *dvh = dv + bh * N * d;
        double *s = (double *)malloc((size_t)N * sizeof(double));
        double *p = (double *)malloc((size_t)N * sizeof(double));
        double *dp = (double *)malloc((size_t)N * sizeof(double));
        if (!s || !p || !dp) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            free(s);
            free(p);
            free(dp);
            continue;
        }
        for (int64_t x = 0; x < N * d; ++x) dkh[x] = dvh[x] = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            score_row_fmt(qh + i * d, kh, i, N, d, scale, causal, fmt, s);
            oracle_safe_softmax(s, N, NULL, p, NULL, NULL);
            double pdp = 0.0; /* sum_k P_ik dP_ik */
            for (int64_t j = 0; j < N; ++j) {
                double acc = 0.0;
                for (int64_t t = 0; t < d; ++t)
                    acc += widen(doh[i * d + t], fmt) * widen(vh[j * d + t], fmt);
                dp[j] = acc;
                pdp += p[j] * acc;
            }
            for (int64_t t = 0; t < d; ++t) dqh[i * d + t] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                if (p[j] == 0.0) continue; /* masked: P = 0 and dS = 0 */
                double ds = p[j] * (dp[j] - pdp);
                for (int64_t t = 0; t < d; ++t) {
                    dvh[j * d + t] += p[j] * widen(doh[i * d + t], fmt);
                    dqh[i * d + t] += scale * ds * widen(kh[j * d + t], fmt);
                    dkh[j * d + t] += scale * ds * widen(qh[i * d + t], fmt);
                }
            }
        }
        free(s);
        free(p);
        free(dp);
    }
    return failed ? -2 : 0;
}

/* oracle_attention_rect_fmt on bf16 inputs. */
int oracle_attention_rect(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int causal,
                          double scale, const int64_t *rows, int64_t n_rows,
                          double *o_out, double *lse_out, double *p_out, int n_threads)
{
    return oracle_attention_rect_fmt(q, k, v, BH, Nq, Nk, d, causal, scale, rows, n_rows,
                                     o_out, lse_out, p_out, n_threads, ORACLE_BF16);
}

/*
 * Square self-attention (Nq == Nk == N): the same computation.
 *   q, k, v : [BH][N][d] bf16 bit patterns
 *   rows    : n_rows query indices (each in [0, N)), applied to every slice;
 *             NULL means all rows (n_rows must then equal N)
 *   o_out   : [BH][n_rows][d] fp64,   O_i = sum_j P_ij v_j
 *   lse_out : [BH][n_rows]   fp64,   LSE_i = m_i + ln(l_i)
 *   p_out   : optional [BH][n_rows][N] fp64 probabilities (may be NULL)
 * Returns 0, or -1 on bad arguments / -2 on allocation failure.
 */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t BH, int64_t N, int64_t d, int causal,
                     double scale, const int64_t *rows, int64_t n_rows,
                     double *o_out, double *lse_out, double *p_out,
                     int n_threads)
{
    return oracle_attention_rect(q, k, v, BH, N, N, d, causal, scale, rows, n_rows,
                                 o_out, lse_out, p_out, n_threads);
}

/* Threads OpenMP would use by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
