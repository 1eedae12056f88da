/*
 * Attention oracle: plain, slow, FP64 CPU reference for the flash-attention
 * forward/backward in its three numerical modes, plus a BF16-rounding
 * emulation of the tiled forward.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, no
 * header and no constant with the CUDA path.
 *
 * Source: "Why Low-Precision Transformer Training Fails: An Analysis on Flash
 * Attention" (arXiv 2510.04212), as summarised on the pages
 *   - section 3.4.4, equation for the safe softmax: P = exp(S - rowmax S),
 *     Obar = P V, O = Obar / rowsum(P);
 *   - section 3.4.5, the stabilised safe softmax: rm = rowmax(S),
 *     rs = rowsum(rm - S <= eps), m' = beta*rm if (rm > 0 and rs > 1) else rm,
 *     m = 0 if (rm < 0 and rs > 1) else m', P = exp(S - m); shift invariance
 *     ("Mathematical equivalence in exact arithmetic");
 *   - section 3.4.2 / 3.4.3: delta = rowsum(dO o O), dS = alpha P o (dP - delta),
 *     dP = dO V^T, dQ = dS K.  dK = dS^T Q and dV = P^T dO are the textbook
 *     gradients of O = softmax(alpha Q K^T) V (the pages state only dQ);
 *   - section 3.4.4, "Concrete bit-level example": BF16 round-to-nearest-even.
 *
 * Readings of the pages used here:
 *   - eps = 0 (the default): a tie is exact equality of raw scores q.k; with
 *     eps > 0 (the exact forward only) keys whose scaled score lies within eps
 *     of the scaled row maximum, alpha*(rm - s) <= eps, count toward rs, over
 *     the whole row as the section's untiled rule states;
 *   - scores are scaled by alpha > 0 before the exponential; the shift rule is
 *     applied to the scaled scores (the sign tests do not depend on alpha > 0);
 *   - causal: key j is visible to query i iff j <= i;
 *   - LSE is the natural log of sum_j exp(alpha s_ij) over visible keys.
 *
 * Arrays are float (holding BF16 values exactly) in [BH][N][d] layout; all
 * arithmetic is double.  Rows are flat indices bh*N + i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- scores ------------------------------------------------------------ */

/* Raw score s = q . k, summed left to right in double.  Products of two BF16
 * values are exact in double; the sum of d <= 256 of them is within a few
 * double ulps of the exact value, and identical key rows give identical
 * scores, so exact ties stay exact. */
static double score(const float* q, const float* k, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += (double)q[c] * (double)k[c];
    return s;
}

static int n_visible(int i, int N, int causal) { return causal ? i + 1 : N; }

static float bf16_round(float x);  /* round to nearest even BF16 (defined below) */

/* Shift for one row in scaled units (section 3.4.5).  rmz = alpha * rowmax,
 * rs = number of keys at the maximum. */
static double row_shift(double rmz, long rs, int mode, double beta) {
    double m = rmz;
    if (mode == 1 && rs > 1) {
        if (rmz > 0.0) m = beta * rmz;
        else if (rmz < 0.0) m = 0.0;
    }
    return m;
}

/* The shift rule alone, exported so tests can check each branch. */
double oracle_row_shift(double rmz, long rs, int mode, double beta) {
    return row_shift(rmz, rs, mode, beta);
}

/* Forward for one row: O row, LSE, tie count; s is scratch of length N. */
static void fwd_row(const float* q, const float* k, const float* v, int N, int d, int i,
                    int causal, double alpha, int mode, double beta, double eps, double* s,
                    double* o, double* lse, int32_t* ties) {
    int nv = n_visible(i, N, causal);
    double rm = -INFINITY;
    for (int j = 0; j < nv; ++j) {
        s[j] = score(q + (size_t)i * d, k + (size_t)j * d, d);
        if (s[j] > rm) rm = s[j];
    }
    long rs = 0;
    for (int j = 0; j < nv; ++j) rs += (eps == 0.0) ? (s[j] == rm) : (alpha * (rm - s[j]) <= eps);
    double m = row_shift(alpha * rm, rs, mode, beta);
    double l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < nv; ++j) {
        double p = exp(alpha * s[j] - m);               /* Pbar = exp(S - m) */
        l += p;                                          /* rowsum(Pbar)      */
        const float* vj = v + (size_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += p * (double)vj[c];   /* Obar = Pbar V */
    }
    for (int c = 0; c < d; ++c) o[c] /= l;              /* O = Obar / rowsum */
    if (lse) *lse = m + log(l);
    if (ties) *ties = (int32_t)rs;
}

/* Forward on selected rows (rows == NULL: all BH*N rows).  Outputs are packed
 * in the order of rows: o[nrows][d], lse[nrows], ties[nrows]; if dout is given,
 * delta[r] = sum_c dO[r,c] * O[r,c] (the backward's rowsum(dO o O)). */
int oracle_fwd(const float* q, const float* k, const float* v, const float* dout,
               int64_t BH, int N, int d, int causal, double alpha, int mode, double beta,
               double eps, const int64_t* rows, int64_t nrows,
               double* o, double* lse, int32_t* ties, double* delta) {
    if (!rows) nrows = BH * (int64_t)N;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            int64_t flat = rows ? rows[r] : r;
            int64_t bh = flat / N;
            int i = (int)(flat % N);
            const size_t off = (size_t)bh * N * d;
            fwd_row(q + off, k + off, v + off, N, d, i, causal, alpha, mode, beta, eps, s,
                    o + (size_t)r * d, lse ? lse + r : NULL, ties ? ties + r : NULL);
            if (dout && delta) {
                const float* g = dout + off + (size_t)i * d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += (double)g[c] * o[(size_t)r * d + c];
                delta[r] = acc;
            }
        }
        free(s);
    }
    return err;
}

/* ---- decomposition of the delta error --------------------------------------
 * For a stored output o of a mode, split delta_lp - delta_hp = sum_c dO[c] *
 * (o[c] - O_hp[c]) (section 3.4.4, "Cause 2: Biased Rounding Error Leads to
 * Positive (delta_lp - delta_hp)[T]") into the quantitative decomposition the
 * page lists as missing: the keys whose BF16 probability is exactly 1, the
 * other keys, and the rounding of the output itself.  With the row's shift m
 * (the untiled rule of the mode with tolerance eps, scaled units),
 *   P_j = fp32(exp(alpha s_j - m)),  b_j = bf16(P_j),  l = sum_j P_j,
 *   p_j = exp(alpha s_j - LSE)        (exact probabilities, O_hp = sum p_j v_j)
 *   one  = sum_c dO[c] sum_{j: b_j = 1}  (b_j / l - p_j) v_j[c]
 *   rest = sum_c dO[c] sum_{j: b_j != 1} (b_j / l - p_j) v_j[c]
 *   out  = sum_c dO[c] (o[c] - sum_j b_j v_j[c] / l)
 * so that one + rest + out = sum_c dO[c] (o[c] - O_hp[c]). */
int oracle_delta_split(const float* q, const float* k, const float* v, const float* o,
                       const float* dout, int64_t BH, int N, int d, int causal, double alpha,
                       int mode, double beta, double eps, const int64_t* rows, int64_t nrows,
                       double* one, double* rest, double* out) {
    if (!rows) nrows = BH * (int64_t)N;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        double* acc = (double*)malloc(sizeof(double) * 5 * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s || !acc) continue;
            int64_t flat = rows ? rows[r] : r;
            int64_t bh = flat / N;
            int i = (int)(flat % N);
            const size_t off = (size_t)bh * N * d;
            const float* qi = q + off + (size_t)i * d;
            int nv = n_visible(i, N, causal);
            double rm = -INFINITY;
            for (int j = 0; j < nv; ++j) {
                s[j] = score(qi, k + off + (size_t)j * d, d);
                if (s[j] > rm) rm = s[j];
            }
            long rs = 0;
            for (int j = 0; j < nv; ++j) rs += (eps == 0.0) ? (s[j] == rm) : (alpha * (rm - s[j]) <= eps);
            double m = row_shift(alpha * rm, rs, mode, beta);
            double lref = 0.0, l = 0.0;
            for (int j = 0; j < nv; ++j) {
                lref += exp(alpha * (s[j] - rm));
                l += (double)(float)exp(alpha * s[j] - m);
            }
            /* acc: [0] sum_{b=1} b v, [1] sum_{b=1} p v, [2] sum_{b!=1} b v, [3] sum_{b!=1} p v */
            for (int c = 0; c < 4 * d; ++c) acc[c] = 0.0;
            for (int j = 0; j < nv; ++j) {
                float pj32 = (float)exp(alpha * s[j] - m);
                double b = (double)bf16_round(pj32);
                double pr = exp(alpha * (s[j] - rm)) / lref;
                const float* vj = v + off + (size_t)j * d;
                int base = (b == 1.0) ? 0 : 2;
                for (int c = 0; c < d; ++c) {
                    acc[(size_t)base * d + c] += b * (double)vj[c];
                    acc[(size_t)(base + 1) * d + c] += pr * (double)vj[c];
                }
            }
            const float* g = dout + off + (size_t)i * d;
            const float* oi = o + off + (size_t)i * d;
            double e1 = 0.0, e2 = 0.0, e3 = 0.0;
            for (int c = 0; c < d; ++c) {
                double one_c = acc[c] / l - acc[(size_t)d + c];
                double rest_c = acc[(size_t)2 * d + c] / l - acc[(size_t)3 * d + c];
                double lp_c = (acc[c] + acc[(size_t)2 * d + c]) / l;
                e1 += (double)g[c] * one_c;
                e2 += (double)g[c] * rest_c;
                e3 += (double)g[c] * ((double)oi[c] - lp_c);
            }
            one[r] = e1;
            rest[r] = e2;
            out[r] = e3;
        }
        free(s);
        free(acc);
    }
    return err;
}

/* ---- backward ------------------------------------------------------------
 * For one head with its exact LSE and delta (= rowsum(dO o O) from the exact
 * O), the gradients of L = sum(dO o O):
 *   P_ij  = exp(alpha s_ij - LSE_i)
 *   dP_ij = dO_i . v_j
 *   dS_ij = alpha P_ij (dP_ij - delta_i)
 *   dQ_i  = sum_j dS_ij k_j,  dK_j = sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i
 * dQ is formed row by row; dK and dV key by key (the same sums, indexed by
 * their output row). */

/* dQ rows.  lse/delta are per flat row (full [BH*N] arrays). */
int oracle_bwd_dq(const float* q, const float* k, const float* v, const float* dout,
                  const double* lse, const double* delta, int64_t BH, int N, int d,
                  int causal, double alpha, const int64_t* rows, int64_t nrows, double* dq) {
    if (!rows) nrows = BH * (int64_t)N;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int64_t bh = flat / N;
        int i = (int)(flat % N);
        const size_t off = (size_t)bh * N * d;
        const float* qi = q + off + (size_t)i * d;
        const float* gi = dout + off + (size_t)i * d;
        double* out = dq + (size_t)r * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        int nv = n_visible(i, N, causal);
        for (int j = 0; j < nv; ++j) {
            const float* kj = k + off + (size_t)j * d;
            const float* vj = v + off + (size_t)j * d;
            double p = exp(alpha * score(qi, kj, d) - lse[flat]);
            double dp = score(gi, vj, d);
            double ds = alpha * p * (dp - delta[flat]);
            for (int c = 0; c < d; ++c) out[c] += ds * (double)kj[c];
        }
    }
    return 0;
}

/* dK and dV rows for the selected keys (flat key index bh*N + j). */
int oracle_bwd_dkdv(const float* q, const float* k, const float* v, const float* dout,
                    const double* lse, const double* delta, int64_t BH, int N, int d,
                    int causal, double alpha, const int64_t* keys, int64_t nkeys,
                    double* dk, double* dv) {
    if (!keys) nkeys = BH * (int64_t)N;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < nkeys; ++r) {
        int64_t flat = keys ? keys[r] : r;
        int64_t bh = flat / N;
        int j = (int)(flat % N);
        const size_t off = (size_t)bh * N * d;
        const float* kj = k + off + (size_t)j * d;
        const float* vj = v + off + (size_t)j * d;
        double* ok = dk + (size_t)r * d;
        double* ov = dv + (size_t)r * d;
        for (int c = 0; c < d; ++c) { ok[c] = 0.0; ov[c] = 0.0; }
        int i0 = causal ? j : 0;
        for (int i = i0; i < N; ++i) {
            const float* qi = q + off + (size_t)i * d;
            const float* gi = dout + off + (size_t)i * d;
            int64_t fi = bh * (int64_t)N + i;
            double p = exp(alpha * score(qi, kj, d) - lse[fi]);
            double dp = score(gi, vj, d);
            double ds = alpha * p * (dp - delta[fi]);
            for (int c = 0; c < d; ++c) {
                ok[c] += ds * (double)qi[c];
                ov[c] += p * (double)gi[c];
            }
        }
    }
    return 0;
}

/* ---- BF16 rounding -------------------------------------------------------
 * Round an FP32 value to the nearest BF16 value, ties to even (section 3.4.4,
 * "Concrete bit-level example": keep 7 fraction bits; round up when the first
 * dropped bit is 1 and any later dropped bit is 1, or when exactly halfway and
 * the kept last bit is 1). */
static float bf16_round(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) {          /* inf / nan: truncate, keep nan quiet */
        if (u & 0x007FFFFFu) u |= 0x00400000u;
        u &= 0xFFFF0000u;
    } else {
        uint32_t dropped = u & 0xFFFFu;
        uint32_t keep = u >> 16;
        if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u))) keep += 1u;
        u = keep << 16;
    }
    float y;
    memcpy(&y, &u, 4);
    return y;
}

void oracle_bf16_round(const float* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = bf16_round(x[i]);
}

/* ---- BF16-rounding emulation of the tiled forward -------------------------
 * Mirrors the schedule of a tiled flash-attention forward with key tiles of
 * block_n keys (the pages' Algorithm 3 with the stabilised lines applied per
 * key tile, section 3.4.5):
 *   - raw scores rounded to FP32;
 *   - per row a running max M and a running count C of keys equal to M
 *     (C restarts when M grows, grows when a tile's max equals M);
 *   - the shift m is the mode's rule applied to (alpha*M, C) after each tile;
 *     when m changes, the accumulated Obar and l are rescaled by
 *     exp(m_old - m_new);
 *   - Pbar = exp(alpha*s - m) rounded to FP32 and then to BF16; l sums the
 *     FP32 values, Obar sums BF16(Pbar) * v exactly (double);
 *   - O = Obar / l rounded to BF16 (modes 0, 1) or FP32 (mode 2).
 * Counters per row:
 *   p_one0 = number of BF16 Pbar entries equal to 1.0,
 *   p_one1 = number of keys whose final weight (Pbar times later rescale
 *            factors) is exactly 1.0, i.e. ones since the last shift change,
 *   p_amb  = entries whose FP32 Pbar lies within 16 FP32 ulps of the BF16
 *            rounding boundary 1 - 2^-9 (either side may be taken by another
 *            correct exponential),
 *   p_max  = the largest BF16 Pbar entry of the row.
 * A second accumulator rounds the running Obar to BF16 after every addition
 * (FP32 add, then BF16 rounding): the reading of the pages' "lp" cumulative
 * error of section 3.4.4 ("How the error accumulates across token
 * positions"); o_peradd = that accumulator / l, unrounded. */
int oracle_fwd_emul(const float* q, const float* k, const float* v, int64_t BH, int N, int d,
                    int causal, double alpha, int mode, double beta, int block_n,
                    const int64_t* rows, int64_t nrows, double* o_out, double* lse_out,
                    int32_t* p_one0, int32_t* p_one1, int32_t* p_amb, double* o_peradd,
                    float* p_max) {
    if (!rows) nrows = BH * (int64_t)N;
    if (block_n < 1) return 1;
    int err = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        float* accp = (float*)malloc(sizeof(float) * (size_t)d);
        float* s32 = (float*)malloc(sizeof(float) * (size_t)N);
        if (!acc || !accp || !s32) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!acc || !accp || !s32) continue;
            int64_t flat = rows ? rows[r] : r;
            int64_t bh = flat / N;
            int i = (int)(flat % N);
            const size_t off = (size_t)bh * N * d;
            const float* qi = q + off + (size_t)i * d;
            int nv = n_visible(i, N, causal);
            for (int j = 0; j < nv; ++j) s32[j] = (float)score(qi, k + off + (size_t)j * d, d);
            for (int c = 0; c < d; ++c) { acc[c] = 0.0; accp[c] = 0.0f; }
            float M = -INFINITY;
            long C = 0;
            double m = -INFINITY, l = 0.0;
            int32_t ones0 = 0, ones1 = 0, amb = 0;
            float pmax = 0.0f;
            const double lo_edge = 1.0 - ldexp(1.0, -9);
            for (int t0 = 0; t0 < nv; t0 += block_n) {
                int t1 = t0 + block_n < nv ? t0 + block_n : nv;
                float tm = -INFINITY;
                for (int j = t0; j < t1; ++j) if (s32[j] > tm) tm = s32[j];
                long tc = 0;
                for (int j = t0; j < t1; ++j) tc += (s32[j] == tm);
                if (tm > M) { M = tm; C = tc; }
                else if (tm == M) C += tc;
                /* shift rule on FP32 values, as a kernel holding FP32 state would */
                float mz = (float)M;
                if (mode == 1 && C > 1) {
                    if (M > 0.0f) mz = (float)beta * M;
                    else if (M < 0.0f) mz = 0.0f;
                }
                double m_new = alpha * (double)mz;
                if (m_new != m) {
                    if (m != -INFINITY) {
                        double rsc = exp(m - m_new);
                        l *= rsc;
                        for (int c = 0; c < d; ++c) {
                            acc[c] *= rsc;
                            accp[c] = bf16_round((float)((double)accp[c] * rsc));
                        }
                    }
                    m = m_new;
                    ones1 = 0;
                }
                for (int j = t0; j < t1; ++j) {
                    float p32 = (float)exp(alpha * (double)s32[j] - m);
                    float pb = bf16_round(p32);
                    if (pb > pmax) pmax = pb;
                    if (pb == 1.0f) { ++ones0; ++ones1; }
                    if (fabs((double)p32 - lo_edge) <= 16.0 * ldexp(1.0, -24)) ++amb;
                    l += (double)p32;
                    const float* vj = v + off + (size_t)j * d;
                    for (int c = 0; c < d; ++c) {
                        acc[c] += (double)pb * (double)vj[c];
                        float prod = pb * vj[c];              /* exact in FP32 */
                        accp[c] = bf16_round(accp[c] + prod); /* FP32 add, BF16 round */
                    }
                }
            }
            for (int c = 0; c < d; ++c) {
                float oc = (float)(acc[c] / l);
                o_out[(size_t)r * d + c] = (mode == 2) ? (double)oc : (double)bf16_round(oc);
                if (o_peradd) o_peradd[(size_t)r * d + c] = (double)accp[c] / l;
            }
            if (lse_out) lse_out[r] = m + log(l);
            if (p_one0) p_one0[r] = ones0;
            if (p_one1) p_one1[r] = ones1;
            if (p_amb) p_amb[r] = amb;
            if (p_max) p_max[r] = pmax;
        }
        free(acc);
        free(accp);
        free(s32);
    }
    return err;
}
