/*
 * tm2_oracle.c -- plain fp64 CPU oracle for the 2Mamba second-order mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides share is the seeded input generator.
 *
 * Source of every formula: "2Mamba2Furious: Linear in Complexity, Competitive
 * in Accuracy" (Mongaras & Larson, arXiv 2602.17363; paperlayer.ai summary):
 *   - Sec. 3 / Sec. 4: the softplus A-mask (decay log l_t = -softplus(a_t)),
 *   - Sec. 5: the square is applied to the QK inner product, the A-mask is
 *     applied to the squared scores, RMSNorm is replaced by "softmax"
 *     normalisation (read here as o_i = N_i / Z_i with the same weights),
 *   - Sec. 2 ("Softmax as a Recurrent Neural Network"): the second-order
 *     hidden state of size (dh^2, dh),
 *   - Sec. 6: 2Mamba-E, softmax attention whose logits carry the softplus
 *     A-mask (the forgetting-transformer form),
 *   - App. A: recurrent inference with a fixed-size state,
 *   - App. C / C.1: gradients of the attention kernel w.r.t. q, k, v and the
 *     A-mask, with separate row and column axis sums.
 *
 * Everything is written as the plain definition: no chunking, no blocking, no
 * reordering beyond the sums the definition states.  OpenMP only splits the
 * loop over independent outputs.  Layout: (B,H,T,.) row-major; state rows are
 * r = m*d + n (key feature indices m, n), state columns are value features.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x), evaluated without overflow. */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

static double sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

static double dot(const double* x, const double* y, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * y[i];
    return s;
}

/* cumA_t = sum_{u <= t} -softplus(a_u): the running log-decay (Sec. 3, Sec. 5). */
static void running_log_decay(const double* a, long T, double* cumA) {
    double s = 0.0;
    for (long t = 0; t < T; ++t) {
        s -= softplus(a[t]);
        cumA[t] = s;
    }
}

void orc_running_log_decay(const double* a, long n_rows, long T, double* cumA) {
    for (long r = 0; r < n_rows; ++r) running_log_decay(a + r * T, T, cumA + r * T);
}

/* s^order for the two orders of the mixer: 2 (2Mamba, Sec. 5) and 1 (the first-order mixer
   of Mamba-2S, Sec. 4: the score itself under the same A-mask). */
static double score_pow(double s, int order) { return order == 1 ? s : s * s; }
/* d(s^order)/ds */
static double score_pow_grad(double s, int order) { return order == 1 ? 1.0 : 2.0 * s; }

/*
 * Quadratic (parallel) form, Sec. 5 (order 2; order 1 replaces the square by the score):
 *   w_ij = exp(cumA_i - cumA_j) * (q_i . k_j)^2      (j <= i)
 *   N_i  = sum_j w_ij v_j,   Z_i = sum_j w_ij
 * plus, when an initial state is given, the term it contributes through the
 * recurrence: exp(cumA_i) * sum_{m,n} q_i[m] q_i[n] S0[(m,n),:] (and z0 for Z).
 * o_i = N_i / Z_i when normalize (o_i = 0 when Z_i == 0), else o_i = N_i.
 */
void orc_fwd_quadratic(int B, int H, int T, int d, int dv,
                       const double* q, const double* k, const double* v, const double* a,
                       const double* S0, const double* z0, int normalize, int order,
                       double* o, double* Z) {
    long BH = (long)B * H;
    double* cum = (double*)malloc(sizeof(double) * (size_t)(BH * T + 1));
    orc_running_log_decay(a, BH, T, cum);
#pragma omp parallel for collapse(2) schedule(dynamic, 8)
    for (long bh = 0; bh < BH; ++bh) {
        for (long i = 0; i < T; ++i) {
            const double* qi = q + (bh * T + i) * d;
            const double* cb = cum + bh * T;
            double* num = (double*)calloc((size_t)dv, sizeof(double));
            double den = 0.0;
            for (long j = 0; j <= i; ++j) {
                double s = dot(qi, k + (bh * T + j) * d, d);
                double w = exp(cb[i] - cb[j]) * score_pow(s, order);
                den += w;
                const double* vj = v + (bh * T + j) * dv;
                for (int c = 0; c < dv; ++c) num[c] += w * vj[c];
            }
            if (S0 || z0) {
                double e = exp(cb[i]);
                for (int m = 0; m < d; ++m)
                    for (int n = 0; n < d; ++n) {
                        double f = e * qi[m] * qi[n];
                        long r = (long)m * d + n;
                        if (S0)
                            for (int c = 0; c < dv; ++c) num[c] += f * S0[(bh * d * d + r) * dv + c];
                        if (z0) den += f * z0[bh * d * d + r];
                    }
            }
            double* oi = o + (bh * T + i) * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = normalize ? (den != 0.0 ? num[c] / den : 0.0) : num[c];
            if (Z) Z[bh * T + i] = den;
            free(num);
        }
    }
    free(cum);
}

/*
 * Recurrent form with the explicit second-order state (Sec. 2, App. A):
 *   gamma_t = exp(-softplus(a_t))
 *   S_t = gamma_t S_{t-1} + (k_t (x) k_t) v_t^T      S in R^{d^2 x dv}
 *   z_t = gamma_t z_{t-1} + (k_t (x) k_t)            z in R^{d^2}
 *   N_t = (q_t (x) q_t)^T S_t,  Z_t = (q_t (x) q_t)^T z_t
 * S0/z0 (nullable) give the state before token 0; S_final/z_final (nullable)
 * receive the state after token T-1.
 */
void orc_fwd_recurrent(int B, int H, int T, int d, int dv,
                       const double* q, const double* k, const double* v, const double* a,
                       const double* S0, const double* z0, int normalize,
                       double* o, double* Z, double* S_final, double* z_final) {
    long BH = (long)B * H;
    long R = (long)d * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        double* S = (double*)calloc((size_t)(R * dv), sizeof(double));
        double* z = (double*)calloc((size_t)R, sizeof(double));
        double* y = (double*)malloc(sizeof(double) * (size_t)dv);
        if (S0) memcpy(S, S0 + bh * R * dv, sizeof(double) * (size_t)(R * dv));
        if (z0) memcpy(z, z0 + bh * R, sizeof(double) * (size_t)R);
        for (long t = 0; t < T; ++t) {
            const double* qt = q + (bh * T + t) * d;
            const double* kt = k + (bh * T + t) * d;
            const double* vt = v + (bh * T + t) * dv;
            double gamma = exp(-softplus(a[bh * T + t]));
            for (int m = 0; m < d; ++m)
                for (int n = 0; n < d; ++n) {
                    long r = (long)m * d + n;
                    double kk = kt[m] * kt[n];
                    z[r] = gamma * z[r] + kk;
                    for (int c = 0; c < dv; ++c) S[r * dv + c] = gamma * S[r * dv + c] + kk * vt[c];
                }
            double zeta = 0.0;
            for (int c = 0; c < dv; ++c) y[c] = 0.0;
            for (int m = 0; m < d; ++m)
                for (int n = 0; n < d; ++n) {
                    long r = (long)m * d + n;
                    double qq = qt[m] * qt[n];
                    zeta += qq * z[r];
                    for (int c = 0; c < dv; ++c) y[c] += qq * S[r * dv + c];
                }
            double* ot = o + (bh * T + t) * dv;
            for (int c = 0; c < dv; ++c)
                ot[c] = normalize ? (zeta != 0.0 ? y[c] / zeta : 0.0) : y[c];
            if (Z) Z[bh * T + t] = zeta;
        }
        if (S_final) memcpy(S_final + bh * R * dv, S, sizeof(double) * (size_t)(R * dv));
        if (z_final) memcpy(z_final + bh * R, z, sizeof(double) * (size_t)R);
        free(S);
        free(z);
        free(y);
    }
}

/*
 * Recurrent form of the first-order mixer (Sec. 2: first-order linear attention keeps a state
 * of size (dh, dh); Sec. 4: Mamba-2S with the softplus A-mask):
 *   S_t = gamma_t S_{t-1} + k_t v_t^T   (d x dv),   z_t = gamma_t z_{t-1} + k_t   (d)
 *   N_t = q_t^T S_t,  Z_t = q_t . z_t,  o_t = N_t / Z_t (normalised) or N_t.
 */
void orc_fwd1_recurrent(int B, int H, int T, int d, int dv,
                        const double* q, const double* k, const double* v, const double* a,
                        int normalize, double* o, double* Z) {
    long BH = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        double* S = (double*)calloc((size_t)(d * dv), sizeof(double));
        double* z = (double*)calloc((size_t)d, sizeof(double));
        for (long t = 0; t < T; ++t) {
            const double* qt = q + (bh * T + t) * d;
            const double* kt = k + (bh * T + t) * d;
            const double* vt = v + (bh * T + t) * dv;
            double gamma = exp(-softplus(a[bh * T + t]));
            for (int m = 0; m < d; ++m) {
                z[m] = gamma * z[m] + kt[m];
                for (int c = 0; c < dv; ++c) S[m * dv + c] = gamma * S[m * dv + c] + kt[m] * vt[c];
            }
            double zeta = dot(qt, z, d);
            double* ot = o + (bh * T + t) * dv;
            for (int c = 0; c < dv; ++c) {
                double y = 0.0;
                for (int m = 0; m < d; ++m) y += qt[m] * S[m * dv + c];
                ot[c] = normalize ? (zeta != 0.0 ? y / zeta : 0.0) : y;
            }
            if (Z) Z[bh * T + t] = zeta;
        }
        free(S);
        free(z);
    }
}

/*
 * One recurrent decode step for N sequences x H heads, in place (App. A):
 * the same update and readout as orc_fwd_recurrent for a single token.
 * q,k: (N,H,d); v: (N,H,dv); a: (N,H); S: (N,H,d*d,dv); z: (N,H,d*d) or NULL.
 * o: (N,H,dv) = y, or y / zeta when normalize (needs z); zeta: (N,H) or NULL.
 */
void orc_step(int N, int H, int d, int dv,
              const double* q, const double* k, const double* v, const double* a,
              double* S, double* z, int normalize, double* o, double* zeta) {
    long NH = (long)N * H;
    long R = (long)d * d;
#pragma omp parallel for schedule(static)
    for (long s = 0; s < NH; ++s) {
        const double* qs = q + s * d;
        const double* ks = k + s * d;
        const double* vs = v + s * dv;
        double gamma = exp(-softplus(a[s]));
        double* Ss = S + s * R * dv;
        double* zs = z ? z + s * R : NULL;
        double y[1024];
        double ze = 0.0;
        for (int c = 0; c < dv; ++c) y[c] = 0.0;
        for (int m = 0; m < d; ++m)
            for (int n = 0; n < d; ++n) {
                long r = (long)m * d + n;
                double kk = ks[m] * ks[n];
                double qq = qs[m] * qs[n];
                for (int c = 0; c < dv; ++c) {
                    Ss[r * dv + c] = gamma * Ss[r * dv + c] + kk * vs[c];
                    y[c] += qq * Ss[r * dv + c];
                }
                if (zs) {
                    zs[r] = gamma * zs[r] + kk;
                    ze += qq * zs[r];
                }
            }
        for (int c = 0; c < dv; ++c)
            o[s * dv + c] = normalize ? (ze != 0.0 ? y[c] / ze : 0.0) : y[c];
        if (zeta) zeta[s] = ze;
    }
}

/*
 * Backward of the quadratic form (App. C / C.1), by the chain rule applied to
 * the definition above with no initial state.  For one (b,h):
 *   upstream: dN_i, dZ_i   (normalised: dN_i = dO_i / Z_i, dZ_i = -(dO_i . o_i) / Z_i;
 *                           unnormalised: dN_i = dO_i, dZ_i = 0)
 *   dw_ij = dN_i . v_j + dZ_i                      gradient into weight w_ij
 *   dv_j  = sum_{i >= j} w_ij dN_i
 *   ds_ij = 2 s_ij exp(cumA_i - cumA_j) dw_ij      s_ij = q_i . k_j  (order 1: exp(..) dw_ij)
 *   dq_i  = sum_{j <= i} ds_ij k_j,   dk_j = sum_{i >= j} ds_ij q_i
 *   dcumA_t = sum_{j <= t} w_tj dw_tj  -  sum_{i >= t} w_it dw_it
 *             (row-axis sum minus column-axis sum, the two A-mask axis sums)
 *   dl_u = sum_{t >= u} dcumA_t       (cumA_t = sum_{u <= t} l_u)
 *   da_u = dl_u * dl_u/da_u = -sigmoid(a_u) * dl_u
 */
void orc_bwd_quadratic(int B, int H, int T, int d, int dv,
                       const double* q, const double* k, const double* v, const double* a,
                       const double* dO, int normalize, int order, const double* o_in, const double* Z_in,
                       double* dq, double* dk, double* dvv, double* da) {
    long BH = (long)B * H;
    for (long bh = 0; bh < BH; ++bh) {
        const double* qb = q + bh * T * d;
        const double* kb = k + bh * T * d;
        const double* vb = v + bh * T * dv;
        const double* ab = a + bh * T;
        const double* gb = dO + bh * T * dv;
        double* cum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* o = (double*)malloc(sizeof(double) * (size_t)(T * dv + 1));
        double* Zs = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* dN = (double*)malloc(sizeof(double) * (size_t)(T * dv + 1));
        double* dZ = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* rowsum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* colsum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        running_log_decay(ab, T, cum);
        /* forward values of this head: recomputed, or (o_in, Z_in non-NULL) the ones the caller
           gives -- the backward of the kernel boundary takes o and Z as inputs (App. C), and with
           given values it is that function of them */
        if (o_in && Z_in) {
            memcpy(o, o_in + bh * T * dv, sizeof(double) * (size_t)(T * dv));
            memcpy(Zs, Z_in + bh * T, sizeof(double) * (size_t)T);
        } else {
            orc_fwd_quadratic(1, 1, T, d, dv, qb, kb, vb, ab, NULL, NULL, normalize, order, o, Zs);
        }
        for (long i = 0; i < T; ++i) {
            if (normalize) {
                double zi = Zs[i];
                double D = dot(gb + i * dv, o + i * dv, dv);
                for (int c = 0; c < dv; ++c) dN[i * dv + c] = zi != 0.0 ? gb[i * dv + c] / zi : 0.0;
                dZ[i] = zi != 0.0 ? -D / zi : 0.0;
            } else {
                for (int c = 0; c < dv; ++c) dN[i * dv + c] = gb[i * dv + c];
                dZ[i] = 0.0;
            }
        }
        /* row-axis quantities: dq_i and sum_j w_ij dw_ij */
#pragma omp parallel for schedule(dynamic, 8)
        for (long i = 0; i < T; ++i) {
            double* dqi = dq + (bh * T + i) * d;
            for (int m = 0; m < d; ++m) dqi[m] = 0.0;
            double rs = 0.0;
            for (long j = 0; j <= i; ++j) {
                double s = dot(qb + i * d, kb + j * d, d);
                double e = exp(cum[i] - cum[j]);
                double w = e * score_pow(s, order);
                double dw = dot(dN + i * dv, vb + j * dv, dv) + dZ[i];
                double ds = score_pow_grad(s, order) * e * dw;
                for (int m = 0; m < d; ++m) dqi[m] += ds * kb[j * d + m];
                rs += w * dw;
            }
            rowsum[i] = rs;
        }
        /* column-axis quantities: dk_j, dv_j and sum_i w_ij dw_ij */
#pragma omp parallel for schedule(dynamic, 8)
        for (long j = 0; j < T; ++j) {
            double* dkj = dk + (bh * T + j) * d;
            double* dvj = dvv + (bh * T + j) * dv;
            for (int m = 0; m < d; ++m) dkj[m] = 0.0;
            for (int c = 0; c < dv; ++c) dvj[c] = 0.0;
            double cs = 0.0;
            for (long i = j; i < T; ++i) {
                double s = dot(qb + i * d, kb + j * d, d);
                double e = exp(cum[i] - cum[j]);
                double w = e * score_pow(s, order);
                double dw = dot(dN + i * dv, vb + j * dv, dv) + dZ[i];
                double ds = score_pow_grad(s, order) * e * dw;
                for (int m = 0; m < d; ++m) dkj[m] += ds * qb[i * d + m];
                for (int c = 0; c < dv; ++c) dvj[c] += w * dN[i * dv + c];
                cs += w * dw;
            }
            colsum[j] = cs;
        }
        double acc = 0.0;
        for (long u = T - 1; u >= 0; --u) {
            acc += rowsum[u] - colsum[u];
            da[bh * T + u] = -sigmoid(ab[u]) * acc;
        }
        free(cum); free(o); free(Zs); free(dN); free(dZ); free(rowsum); free(colsum);
    }
}

/*
 * 2Mamba-E forward (Sec. 6): softmax attention whose logits carry the A-mask,
 *   x_ij = scale * (q_i . k_j) + cumA_i - cumA_j     (j <= i)
 *   o_i  = sum_j softmax_j(x_i.) v_j,   lse_i = log sum_j exp(x_ij)
 * evaluated in two passes (true row maximum first), not with an online max.
 */
void orc_e_fwd(int B, int H, int T, int d, int dv,
               const double* q, const double* k, const double* v, const double* a,
               double scale, double* o, double* lse) {
    long BH = (long)B * H;
    double* cum = (double*)malloc(sizeof(double) * (size_t)(BH * T + 1));
    orc_running_log_decay(a, BH, T, cum);
#pragma omp parallel for collapse(2) schedule(dynamic, 8)
    for (long bh = 0; bh < BH; ++bh) {
        for (long i = 0; i < T; ++i) {
            const double* cb = cum + bh * T;
            const double* qi = q + (bh * T + i) * d;
            double mx = -INFINITY;
            for (long j = 0; j <= i; ++j) {
                double x = scale * dot(qi, k + (bh * T + j) * d, d) + cb[i] - cb[j];
                if (x > mx) mx = x;
            }
            double sum = 0.0;
            double* oi = o + (bh * T + i) * dv;
            for (int c = 0; c < dv; ++c) oi[c] = 0.0;
            for (long j = 0; j <= i; ++j) {
                double x = scale * dot(qi, k + (bh * T + j) * d, d) + cb[i] - cb[j];
                double p = exp(x - mx);
                sum += p;
                const double* vj = v + (bh * T + j) * dv;
                for (int c = 0; c < dv; ++c) oi[c] += p * vj[c];
            }
            for (int c = 0; c < dv; ++c) oi[c] /= sum;
            if (lse) lse[bh * T + i] = mx + log(sum);
        }
    }
    free(cum);
}

/*
 * 2Mamba-E backward (Sec. 6 with App. C): with P_ij = exp(x_ij - lse_i),
 *   D_i = dO_i . o_i,  dx_ij = P_ij (dO_i . v_j - D_i)
 *   dv_j = sum_{i >= j} P_ij dO_i
 *   dq_i = scale * sum_{j <= i} dx_ij k_j,  dk_j = scale * sum_{i >= j} dx_ij q_i
 *   dcumA_t = sum_{j <= t} dx_tj - sum_{i >= t} dx_it,  da_u = -sigmoid(a_u) sum_{t >= u} dcumA_t
 */
void orc_e_bwd(int B, int H, int T, int d, int dv,
               const double* q, const double* k, const double* v, const double* a,
               const double* dO, double scale,
               double* dq, double* dk, double* dvv, double* da) {
    long BH = (long)B * H;
    for (long bh = 0; bh < BH; ++bh) {
        const double* qb = q + bh * T * d;
        const double* kb = k + bh * T * d;
        const double* vb = v + bh * T * dv;
        const double* ab = a + bh * T;
        const double* gb = dO + bh * T * dv;
        double* cum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* o = (double*)malloc(sizeof(double) * (size_t)(T * dv + 1));
        double* lse = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* D = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* rowsum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        double* colsum = (double*)malloc(sizeof(double) * (size_t)(T + 1));
        running_log_decay(ab, T, cum);
        orc_e_fwd(1, 1, T, d, dv, qb, kb, vb, ab, scale, o, lse);
        for (long i = 0; i < T; ++i) D[i] = dot(gb + i * dv, o + i * dv, dv);
#pragma omp parallel for schedule(dynamic, 8)
        for (long i = 0; i < T; ++i) {
            double* dqi = dq + (bh * T + i) * d;
            for (int m = 0; m < d; ++m) dqi[m] = 0.0;
            double rs = 0.0;
            for (long j = 0; j <= i; ++j) {
                double x = scale * dot(qb + i * d, kb + j * d, d) + cum[i] - cum[j];
                double p = exp(x - lse[i]);
                double dx = p * (dot(gb + i * dv, vb + j * dv, dv) - D[i]);
                for (int m = 0; m < d; ++m) dqi[m] += scale * dx * kb[j * d + m];
                rs += dx;
            }
            rowsum[i] = rs;
        }
#pragma omp parallel for schedule(dynamic, 8)
        for (long j = 0; j < T; ++j) {
            double* dkj = dk + (bh * T + j) * d;
            double* dvj = dvv + (bh * T + j) * dv;
            for (int m = 0; m < d; ++m) dkj[m] = 0.0;
            for (int c = 0; c < dv; ++c) dvj[c] = 0.0;
            double cs = 0.0;
            for (long i = j; i < T; ++i) {
                double x = scale * dot(qb + i * d, kb + j * d, d) + cum[i] - cum[j];
                double p = exp(x - lse[i]);
                double dx = p * (dot(gb + i * dv, vb + j * dv, dv) - D[i]);
                for (int m = 0; m < d; ++m) dkj[m] += scale * dx * qb[i * d + m];
                for (int c = 0; c < dv; ++c) dvj[c] += p * gb[i * dv + c];
                cs += dx;
            }
            colsum[j] = cs;
        }
        double acc = 0.0;
        for (long u = T - 1; u >= 0; --u) {
            acc += rowsum[u] - colsum[u];
            da[bh * T + u] = -sigmoid(ab[u]) * acc;
        }
        free(cum); free(o); free(lse); free(D); free(rowsum); free(colsum);
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Size-2 causal input convolution of Mamba-2S, kept by 2Mamba (Sec. 3: kernel size 2;
 * Sec. 4: no activation; App. A: inference caches the previous raw token).  Per channel c of
 * head h, a depthwise convolution over time:
 *   y_t[c] = w[h][c][0] x_t[c] + w[h][c][1] x_{t-1}[c] + b[h][c],   x_{-1} = x_prev (or 0).
 * x, y: (B,H,T,C); w: (H,C,2); b: (H,C) or NULL; x_prev: (B,H,C) or NULL.
 */
void orc_conv2_fwd(int B, int H, int T, int C, const double* x, const double* w, const double* b,
                   const double* x_prev, double* y) {
    for (long bb = 0; bb < B; ++bb)
        for (long h = 0; h < H; ++h)
            for (long t = 0; t < T; ++t)
                for (int c = 0; c < C; ++c) {
                    long bh = bb * H + h;
                    double prev = t > 0 ? x[(bh * T + t - 1) * C + c] : (x_prev ? x_prev[bh * C + c] : 0.0);
                    double out = w[(h * C + c) * 2] * x[(bh * T + t) * C + c] + w[(h * C + c) * 2 + 1] * prev;
                    if (b) out += b[h * C + c];
                    y[(bh * T + t) * C + c] = out;
                }
}

/* Its gradients, by the chain rule on the definition above: dx_t gets w0 dy_t from y_t and
 * w1 dy_{t+1} from y_{t+1}; dx_prev = w1 dy_0; dw0, dw1, db sum dy_t x_t, dy_t x_{t-1}, dy_t
 * over every batch row and time step of the head.  dx_prev, db may be NULL. */
void orc_conv2_bwd(int B, int H, int T, int C, const double* x, const double* w, const double* x_prev,
                   const double* dy, double* dx, double* dx_prev, double* dw, double* db) {
    for (long i = 0; i < (long)H * C * 2; ++i) dw[i] = 0.0;
    if (db)
        for (long i = 0; i < (long)H * C; ++i) db[i] = 0.0;
    for (long bb = 0; bb < B; ++bb)
        for (long h = 0; h < H; ++h)
            for (long t = 0; t < T; ++t)
                for (int c = 0; c < C; ++c) {
                    long bh = bb * H + h;
                    double g = dy[(bh * T + t) * C + c];
                    double next = t + 1 < T ? dy[(bh * T + t + 1) * C + c] : 0.0;
                    dx[(bh * T + t) * C + c] = w[(h * C + c) * 2] * g + w[(h * C + c) * 2 + 1] * next;
                    double prev = t > 0 ? x[(bh * T + t - 1) * C + c] : (x_prev ? x_prev[bh * C + c] : 0.0);
                    dw[(h * C + c) * 2] += g * x[(bh * T + t) * C + c];
                    dw[(h * C + c) * 2 + 1] += g * prev;
                    if (db) db[h * C + c] += g;
                    if (t == 0 && dx_prev) dx_prev[bh * C + c] = w[(h * C + c) * 2 + 1] * g;
                }
}
