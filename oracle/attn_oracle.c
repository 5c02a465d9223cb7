/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for the attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference for the
 * CUDA library in tensor_attn_fwd_gb300/.  The two share no code, headers,
 * helpers or constants.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load or call it; the product
 * path never does.
 *
 * What it computes (source: "A Thread-Register Decoupled GPU Execution Model
 * for Efficient Tensor Computation", Background, Equ. 1 -- the multi-head
 * attention that the FlashAttention series computes fused; the equation is
 * referenced there but not printed, so its standard content is written out
 * here):
 *
 *   for every batch b and query head h, with KV head g = h / (Hq / Hkv)
 *   (grouped-query sharing, same page, Methodology: "GQA with eight heads per
 *   group", MQA when Hkv = 1):
 *     s_ij   = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]
 *     vis_ij = (j < Sk) and (not causal or j <= i + Sk - Sq)   (bottom-right)
 *     m_i    = max over visible j of s_ij
 *     e_ij   = exp(s_ij - m_i)            (visible j only)
 *     l_i    = sum_j e_ij
 *     O[i,:] = sum_j e_ij * V[b,g,j,:] / l_i
 *     LSE_i  = m_i + ln(l_i)              (natural log, includes the scale)
 *   A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Decode (same page, Methodology / Evaluation: FlashDecoding -- GEMV plus
 * softmax, memory bound) is the same definition with Sq = 1, no mask, split
 * along the key axis: chunk = ceil(Sk / ns), split s covers keys
 * [s*chunk, min(Sk, (s+1)*chunk)); each split returns its own normalised
 * O_s and its own LSE_s (empty split: O_s = 0, LSE_s = -inf), and the
 * combine step returns LSE = ln sum_s exp(LSE_s) and
 * O = sum_s exp(LSE_s - LSE) * O_s.
 *
 * Inputs are bf16 bit patterns (uint16, row-major [B,H,S,D]); each value is
 * widened exactly to double.  All arithmetic is double, in the order the
 * definition states; there is no blocking, no online softmax and no
 * reordering beyond it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Number of visible keys for query row i: the visible set is the prefix
 * [0, nvis) of the key axis. */
static int64_t visible_keys(int64_t i, int64_t Sq, int64_t Sk, int causal)
{
    if (!causal) return Sk;
    int64_t n = i + Sk - Sq + 1;
    if (n < 0) n = 0;
    if (n > Sk) n = Sk;
    return n;
}

/* One query row against keys [j0, j1) of one KV head.
 * q: D values (double); kh, vh: the KV head's [Sk, D] bf16 matrices.
 * s: scratch of at least (j1 - j0) doubles. */
static void attend_row(const double *q, const uint16_t *kh, const uint16_t *vh,
                       int64_t j0, int64_t j1, int64_t D, double scale,
                       double *s, double *o, double *lse)
{
    int64_t n = j1 - j0;
    if (n <= 0) {
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* scores */
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *kr = kh + (j0 + j) * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += q[d] * bf16_to_double(kr[d]);
        s[j] = scale * acc;
    }
    /* m = max over visible keys */
    double m = s[0];
    for (int64_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    /* e = exp(s - m), l = sum e (e overwrites s) */
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* O = sum e * V / l */
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *vr = vh + (j0 + j) * D;
        double e = s[j];
        for (int64_t d = 0; d < D; ++d) o[d] += e * bf16_to_double(vr[d]);
    }
    for (int64_t d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
}

static int check_dims(int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                      int64_t D)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

/*
 * Attention forward for a list of query rows.
 *   rows: flat row ids r = (b*Hq + h)*Sq + i; NULL means every row in order.
 *   o_out: [nrows, D] doubles; lse_out: [nrows] doubles.
 * Returns 0 on success, nonzero on invalid arguments.
 */
int oracle_attn_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                         int64_t Sk, int64_t D, int causal, double scale,
                         const int64_t *rows, int64_t nrows, double *o_out,
                         double *lse_out)
{
    if (check_dims(B, Hq, Hkv, Sq, Sk, D)) return 1;
    int64_t total = B * Hq * Sq;
    if (rows == NULL) nrows = total;
    int64_t group = Hq / Hkv;
    int bad = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (s == NULL || qd == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < nrows; ++t) {
                int64_t r = rows ? rows[t] : t;
                if (r < 0 || r >= total) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                int64_t i = r % Sq;
                int64_t bh = r / Sq;
                int64_t h = bh % Hq;
                int64_t b = bh / Hq;
                int64_t g = h / group;
                const uint16_t *qr = q + r * D;
                for (int64_t d = 0; d < D; ++d) qd[d] = bf16_to_double(qr[d]);
                const uint16_t *kh = k + (b * Hkv + g) * Sk * D;
                const uint16_t *vh = v + (b * Hkv + g) * Sk * D;
                int64_t nvis = visible_keys(i, Sq, Sk, causal);
                attend_row(qd, kh, vh, 0, nvis, D, scale, s, o_out + t * D,
                           lse_out + t);
            }
        }
        free(s);
        free(qd);
    }
    return bad;
}

/*
 * Split-KV decode partials (Sq = 1, no mask).
 *   q: [B,Hq,1,D]; k, v: [B,Hkv,Sk,D] (bf16 bits).
 *   o_part: [ns,B,Hq,D]; lse_part: [ns,B,Hq].
 *   align >= 1: the chunk ceil(Sk/ns) is rounded up to a multiple of align
 *   (1 = the plain rule; the paged-cache decode splits whole blocks of keys).
 */
int oracle_decode_split(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t Sk, int64_t D,
                        int64_t ns, int64_t align, double scale, double *o_part,
                        double *lse_part)
{
    if (check_dims(B, Hq, Hkv, 1, Sk, D) || ns <= 0 || align <= 0) return 1;
    int64_t group = Hq / Hkv;
    int64_t chunk = (Sk + ns - 1) / ns;
    chunk = (chunk + align - 1) / align * align;
    int64_t units = ns * B * Hq;
    int bad = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(chunk > 0 ? chunk : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (s == NULL || qd == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t u = 0; u < units; ++u) {
                int64_t bh = u % (B * Hq);
                int64_t sp = u / (B * Hq);
                int64_t h = bh % Hq;
                int64_t b = bh / Hq;
                int64_t g = h / group;
                const uint16_t *qr = q + bh * D;
                for (int64_t d = 0; d < D; ++d) qd[d] = bf16_to_double(qr[d]);
                int64_t j0 = sp * chunk;
                int64_t j1 = j0 + chunk;
                if (j0 > Sk) j0 = Sk;
                if (j1 > Sk) j1 = Sk;
                const uint16_t *kh = k + (b * Hkv + g) * Sk * D;
                const uint16_t *vh = v + (b * Hkv + g) * Sk * D;
                attend_row(qd, kh, vh, j0, j1, D, scale, s, o_part + u * D,
                           lse_part + u);
            }
        }
        free(s);
        free(qd);
    }
    return bad;
}

/*
 * Log-sum-exp combine of ns partials.
 *   o_part: [ns,R,D]; lse_part: [ns,R] with R = B*Hq rows.
 *   o: [R,D]; lse: [R].
 */
int oracle_combine(const double *o_part, const double *lse_part, int64_t R,
                   int64_t D, int64_t ns, double *o, double *lse)
{
    if (R < 0 || D <= 0 || ns <= 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        double M = -INFINITY;
        for (int64_t sp = 0; sp < ns; ++sp)
            if (lse_part[sp * R + r] > M) M = lse_part[sp * R + r];
        for (int64_t d = 0; d < D; ++d) o[r * D + d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double W = 0.0;
        for (int64_t sp = 0; sp < ns; ++sp) W += exp(lse_part[sp * R + r] - M);
        double L = M + log(W);
        for (int64_t sp = 0; sp < ns; ++sp) {
            double w = exp(lse_part[sp * R + r] - L);
            if (w == 0.0) continue;
            for (int64_t d = 0; d < D; ++d)
                o[r * D + d] += w * o_part[(sp * R + r) * D + d];
        }
        lse[r] = L;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Attention backward (TEST INFRASTRUCTURE, like everything in this file).
 *
 * The gradient of O = softmax(S) V with S = scale * Q K^T (+ mask) for an
 * upstream gradient dO, written out row by row from the chain rule:
 *   P_ij  = exp(s_ij - LSE_i)                 (visible j only)
 *   dV_j  = sum_i P_ij dO_i                   (summed over the group's heads)
 *   dP_ij = dO_i . V_j
 *   Delta_i = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i           (summed over the group's heads)
 * Inputs are doubles here (the Python side widens bf16 exactly), so that a
 * finite-difference check can perturb them.
 * ------------------------------------------------------------------------ */

/* Forward on double inputs (same definition as oracle_attn_fwd_rows). */
int oracle_attn_fwd_f64(const double *q, const double *k, const double *v, int64_t B,
                        int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D, int causal,
                        double scale, double *o, double *lse)
{
    if (check_dims(B, Hq, Hkv, Sq, Sk, D)) return 1;
    int64_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        if (s == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < B * Hq * Sq; ++r) {
                int64_t i = r % Sq, bh = r / Sq, h = bh % Hq, b = bh / Hq;
                int64_t g = h / group;
                const double *qr = q + r * D;
                const double *kh = k + (b * Hkv + g) * Sk * D;
                const double *vh = v + (b * Hkv + g) * Sk * D;
                int64_t n = visible_keys(i, Sq, Sk, causal);
                double *orow = o + r * D;
                if (n <= 0) {
                    for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
                    lse[r] = -INFINITY;
                    continue;
                }
                for (int64_t j = 0; j < n; ++j) {
                    double acc = 0.0;
                    for (int64_t d = 0; d < D; ++d) acc += qr[d] * kh[j * D + d];
                    s[j] = scale * acc;
                }
                double m = s[0];
                for (int64_t j = 1; j < n; ++j)
                    if (s[j] > m) m = s[j];
                double l = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    s[j] = exp(s[j] - m);
                    l += s[j];
                }
                for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
                for (int64_t j = 0; j < n; ++j)
                    for (int64_t d = 0; d < D; ++d) orow[d] += s[j] * vh[j * D + d];
                for (int64_t d = 0; d < D; ++d) orow[d] /= l;
                lse[r] = m + log(l);
            }
        }
        free(s);
    }
    return bad;
}

/* Backward.  q, dO: [B,Hq,Sq,D]; k, v: [B,Hkv,Sk,D] (doubles).
 * dq: [B,Hq,Sq,D]; dk, dv: [B,Hkv,Sk,D] (overwritten). */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *dout,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                        int causal, double scale, double *dq, double *dk, double *dv)
{
    if (check_dims(B, Hq, Hkv, Sq, Sk, D)) return 1;
    int64_t group = Hq / Hkv;
    int bad = 0;
    for (int64_t t = 0; t < B * Hkv * Sk * D; ++t) {
        dk[t] = 0.0;
        dv[t] = 0.0;
    }
    /* One KV head per task: its dK/dV rows are owned by exactly one thread. */
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        if (p == NULL || dp == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bg = 0; bg < B * Hkv; ++bg) {
                int64_t b = bg / Hkv, g = bg % Hkv;
                const double *kh = k + bg * Sk * D;
                const double *vh = v + bg * Sk * D;
                double *dkh = dk + bg * Sk * D;
                double *dvh = dv + bg * Sk * D;
                for (int64_t h = g * group; h < (g + 1) * group; ++h) {
                    int64_t bh = b * Hq + h;
                    for (int64_t i = 0; i < Sq; ++i) {
                        const double *qr = q + (bh * Sq + i) * D;
                        const double *dor = dout + (bh * Sq + i) * D;
                        double *dqr = dq + (bh * Sq + i) * D;
                        for (int64_t d = 0; d < D; ++d) dqr[d] = 0.0;
                        int64_t n = visible_keys(i, Sq, Sk, causal);
                        if (n <= 0) continue;
                        /* P row */
                        for (int64_t j = 0; j < n; ++j) {
                            double acc = 0.0;
                            for (int64_t d = 0; d < D; ++d) acc += qr[d] * kh[j * D + d];
                            p[j] = scale * acc;
                        }
                        double m = p[0];
                        for (int64_t j = 1; j < n; ++j)
                            if (p[j] > m) m = p[j];
                        double l = 0.0;
                        for (int64_t j = 0; j < n; ++j) {
                            p[j] = exp(p[j] - m);
                            l += p[j];
                        }
                        for (int64_t j = 0; j < n; ++j) p[j] /= l;
                        /* dP row and Delta */
                        double delta = 0.0;
                        for (int64_t j = 0; j < n; ++j) {
                            double acc = 0.0;
                            for (int64_t d = 0; d < D; ++d) acc += dor[d] * vh[j * D + d];
                            dp[j] = acc;
                            delta += p[j] * acc;
                        }
                        /* dS and the three products */
                        for (int64_t j = 0; j < n; ++j) {
                            double ds = p[j] * (dp[j] - delta);
                            for (int64_t d = 0; d < D; ++d) {
                                dqr[d] += scale * ds * kh[j * D + d];
                                dkh[j * D + d] += scale * ds * qr[d];
                                dvh[j * D + d] += p[j] * dor[d];
                            }
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return bad;
}

/* ------------------------------------------------------------------------
 * Backward at sampled positions, on bf16 inputs, for problems too large for
 * oracle_attn_bwd_f64.  Same definitions as above:
 *   dq_out[r]  = dQ of query row qrows[r]   (flat (b*Hq + h)*Sq + i)
 *   dk_out[t], dv_out[t] = dK, dV of key keys[t]   (flat (b*Hkv + g)*Sk + j)
 * A key's gradient needs LSE_i and Delta_i of every row i of the group's
 * heads, so those are computed first for each (b, g) that a sampled key
 * belongs to (one full row pass each); then each key sums over those rows.
 * ------------------------------------------------------------------------ */

/* P (normalised), dP and Delta of one query row against its visible keys.
 * p, dp: scratch of at least Sk doubles.  Returns the number of visible keys. */
static int64_t bwd_row_bf16(const uint16_t *qr, const uint16_t *dor, const uint16_t *kh,
                            const uint16_t *vh, int64_t n, int64_t D, double scale,
                            double *p, double *dp, double *lse_out, double *delta_out)
{
    if (n <= 0) {
        *lse_out = -INFINITY;
        *delta_out = 0.0;
        return 0;
    }
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d)
            acc += bf16_to_double(qr[d]) * bf16_to_double(kh[j * D + d]);
        p[j] = scale * acc;
    }
    double m = p[0];
    for (int64_t j = 1; j < n; ++j)
        if (p[j] > m) m = p[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int64_t j = 0; j < n; ++j) p[j] /= l;
    double delta = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d)
            acc += bf16_to_double(dor[d]) * bf16_to_double(vh[j * D + d]);
        dp[j] = acc;
        delta += p[j] * acc;
    }
    *lse_out = m + log(l);
    *delta_out = delta;
    return n;
}

int oracle_attn_bwd_sampled(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const uint16_t *dout, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t Sq, int64_t Sk, int64_t D, int causal, double scale,
                            const int64_t *qrows, int64_t nq, const int64_t *keys, int64_t nk,
                            double *dq_out, double *dk_out, double *dv_out)
{
    if (check_dims(B, Hq, Hkv, Sq, Sk, D)) return 1;
    for (int64_t r = 0; r < nq; ++r)
        if (qrows[r] < 0 || qrows[r] >= B * Hq * Sq) return 1;
    for (int64_t t = 0; t < nk; ++t)
        if (keys[t] < 0 || keys[t] >= B * Hkv * Sk) return 1;
    int64_t group = Hq / Hkv;
    int bad = 0;

    /* dQ rows */
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        if (p == NULL || dp == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < nq; ++r) {
                int64_t row = qrows[r];
                int64_t i = row % Sq, bh = row / Sq, h = bh % Hq, b = bh / Hq;
                int64_t bg = b * Hkv + h / group;
                const uint16_t *kh = k + bg * Sk * D, *vh = v + bg * Sk * D;
                double lse, delta;
                int64_t n = bwd_row_bf16(q + row * D, dout + row * D, kh, vh,
                                         visible_keys(i, Sq, Sk, causal), D, scale, p, dp,
                                         &lse, &delta);
                double *dqr = dq_out + r * D;
                for (int64_t d = 0; d < D; ++d) dqr[d] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    double ds = p[j] * (dp[j] - delta);
                    for (int64_t d = 0; d < D; ++d) dqr[d] += scale * ds * bf16_to_double(kh[j * D + d]);
                }
            }
        }
        free(p);
        free(dp);
    }
    if (bad) return bad;

    /* dK / dV keys, one (b, g) at a time */
    double *lse_g = (double *)malloc(sizeof(double) * (size_t)(group * Sq > 0 ? group * Sq : 1));
    double *delta_g = (double *)malloc(sizeof(double) * (size_t)(group * Sq > 0 ? group * Sq : 1));
    char *done = (char *)calloc((size_t)(nk > 0 ? nk : 1), 1);
    if (lse_g == NULL || delta_g == NULL || done == NULL) bad = 2;
    for (int64_t t0 = 0; t0 < nk && !bad; ++t0) {
        if (done[t0]) continue;
        int64_t bg = keys[t0] / Sk, b = bg / Hkv, g = bg % Hkv;
        const uint16_t *kh = k + bg * Sk * D, *vh = v + bg * Sk * D;
        /* row statistics of the group's heads */
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
            double *dp = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
            if (p == NULL || dp == NULL) {
#pragma omp atomic write
                bad = 2;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t gr = 0; gr < group * Sq; ++gr) {
                    int64_t h = g * group + gr / Sq, i = gr % Sq;
                    int64_t row = (b * Hq + h) * Sq + i;
                    bwd_row_bf16(q + row * D, dout + row * D, kh, vh,
                                 visible_keys(i, Sq, Sk, causal), D, scale, p, dp,
                                 &lse_g[gr], &delta_g[gr]);
                }
            }
            free(p);
            free(dp);
        }
        if (bad) break;
        /* every sampled key of this (b, g) */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t t = t0; t < nk; ++t) {
            if (keys[t] / Sk != bg) continue;
            done[t] = 1;
            int64_t j = keys[t] % Sk;
            double *dkr = dk_out + t * D, *dvr = dv_out + t * D;
            for (int64_t d = 0; d < D; ++d) {
                dkr[d] = 0.0;
                dvr[d] = 0.0;
            }
            for (int64_t gr = 0; gr < group * Sq; ++gr) {
                int64_t h = g * group + gr / Sq, i = gr % Sq;
                if (j >= visible_keys(i, Sq, Sk, causal)) continue;
                int64_t row = (b * Hq + h) * Sq + i;
                const uint16_t *qr = q + row * D, *dor = dout + row * D;
                double s = 0.0, dpv = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    s += bf16_to_double(qr[d]) * bf16_to_double(kh[j * D + d]);
                    dpv += bf16_to_double(dor[d]) * bf16_to_double(vh[j * D + d]);
                }
                double pij = exp(scale * s - lse_g[gr]);
                double ds = pij * (dpv - delta_g[gr]);
                for (int64_t d = 0; d < D; ++d) {
                    dkr[d] += scale * ds * bf16_to_double(qr[d]);
                    dvr[d] += pij * bf16_to_double(dor[d]);
                }
            }
        }
    }
    free(lse_g);
    free(delta_g);
    free(done);
    return bad;
}

/* ------------------------------------------------------------------------
 * QKV projection + rotary position embedding, in front of attention.
 * Source: "A Thread-Register Decoupled GPU Execution Model for Efficient
 * Tensor Computation", Background (a linear projection of the hidden states
 * gives Q, K and V, each a GEMM with its weight; RoPE is applied in many
 * architectures) and "VDCores: Resource Decoupled Programming and Execution
 * for Asynchronous GPUs", Evaluation (the QKV-Projection + RoPE fused pattern).
 * The pages print no RoPE formula; the standard rotary embedding is written
 * out here:
 *   y[t][n]   = sum_h x[t][h] * w[n][h]          (w holds the rows of Wq, Wk, Wv)
 *   columns [0, Hq*D) are Q heads, then Hkv K heads, then Hkv V heads;
 *   theta_i   = base^(-2i/D),  angle = pos_t * theta_i,  i in [0, D/2)
 *   style 0 (pairs of adjacent dims):  (a, b) = (y[2i], y[2i+1])
 *   style 1 (dims i and i + D/2):      (a, b) = (y[i], y[i+D/2])
 *   a' = a cos(angle) - b sin(angle),   b' = a sin(angle) + b cos(angle)
 * applied to every Q and K head; V is the plain projection.
 * Outputs for the listed tokens t (t = b*S + s): q [n, Hq, D], k, v [n, Hkv, D].
 * ------------------------------------------------------------------------ */
int oracle_qkv_rope(const uint16_t *x, const uint16_t *w, const int32_t *positions,
                    int64_t T, int64_t hidden, int64_t Hq, int64_t Hkv, int64_t D,
                    double base, int style, const int64_t *tokens, int64_t ntok,
                    double *q, double *k, double *v)
{
    if (T < 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D % 2 != 0) return 1;
    if (style != 0 && style != 1) return 1;
    for (int64_t r = 0; r < ntok; ++r)
        if (tokens[r] < 0 || tokens[r] >= T) return 1;
    int64_t N = (Hq + 2 * Hkv) * D;
    int bad = 0;
#pragma omp parallel
    {
        double *y = (double *)malloc(sizeof(double) * (size_t)N);
        double *xr = (double *)malloc(sizeof(double) * (size_t)hidden);
        if (y == NULL || xr == NULL) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < ntok; ++r) {
                int64_t t = tokens[r];
                for (int64_t h = 0; h < hidden; ++h) xr[h] = bf16_to_double(x[t * hidden + h]);
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int64_t h = 0; h < hidden; ++h)
                        acc += xr[h] * bf16_to_double(w[n * hidden + h]);
                    y[n] = acc;
                }
                double pos = (double)positions[t];
                /* rotate every Q and K head */
                for (int64_t head = 0; head < Hq + Hkv; ++head) {
                    double *yh = y + head * D;
                    for (int64_t i = 0; i < D / 2; ++i) {
                        double theta = pow(base, -2.0 * (double)i / (double)D);
                        double ang = pos * theta;
                        double c = cos(ang), s = sin(ang);
                        int64_t ia = style == 0 ? 2 * i : i;
                        int64_t ib = style == 0 ? 2 * i + 1 : i + D / 2;
                        double a = yh[ia], b = yh[ib];
                        yh[ia] = a * c - b * s;
                        yh[ib] = a * s + b * c;
                    }
                }
                for (int64_t n = 0; n < Hq * D; ++n) q[r * Hq * D + n] = y[n];
                for (int64_t n = 0; n < Hkv * D; ++n) {
                    k[r * Hkv * D + n] = y[Hq * D + n];
                    v[r * Hkv * D + n] = y[(Hq + Hkv) * D + n];
                }
            }
        }
        free(y);
        free(xr);
    }
    return bad;
}
