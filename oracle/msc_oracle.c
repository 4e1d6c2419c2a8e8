/*
 * msc_oracle.c -- plain double-precision CPU oracle for the Mamba selective scan.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
 * and bench.py's CPU-baseline leg may load or call this file.  It shares no code,
 * header, table or helper with the CUDA library; it is written straight from the
 * pages' definitions, one sequential step at a time, with no blocking, fusion or
 * reordering:
 *
 *   Selection (bqwf survey sec. 2.2; "Mamba 解密" sec. 5):
 *       Delta_t = softplus(delta_t + Delta_bias)
 *   Exponential-Euler discretisation ("Mamba 解密" sec. 6.3: Mamba-1 and
 *   Mamba-2 are exponential-Euler; recurrence of its sec. 3/5 with the Euler input):
 *       abar_{t,n} = exp(Delta_t * A[n])
 *       h_{t,n}    = abar_{t,n} * h_{t-1,n} + Delta_t * B_{t,n} * u_t
 *   Readout with direct feed-through D ("Mamba 解密" sec. 3):
 *       y'_t = sum_n C_{t,n} h_{t,n} + D * u_t
 *   Gate ("Mamba前世今生全挖掘" sec. 二: selective SSM plus gating):  y_t = y'_t * silu(z_t)
 *
 *   SSD (bqwf survey sec. 3.2: scalar A_t = alpha_t I; "Mamba 解密"
 *   sec. 6.2: M_ij = a_{j+1} ... a_i): per head the state is a P x N matrix
 *       H_t = a_t H_{t-1} + Delta_t x_t B_t^T,   y_t = H_t C_t (+ D x_t)(* silu z_t)
 *   which is the S6 recurrence with channels d = (head, p) sharing Delta and A.
 *
 * The backward is hand-derived from the forward (the pages only say that the
 * gradient recomputes states instead of storing them, bqwf survey sec. 2.2):
 *   g'_t = dy_t * silu(z_t)
 *   dz_t = dy_t * y'_t * sig(z_t) * (1 + z_t (1 - sig(z_t)))
 *   lambda_{t,n} = g'_t C_{t,n} + abar_{t+1,n} lambda_{t+1,n}    (lambda_{L} = 0)
 *   dC_{t,n} += g'_t h_{t,n};  dB_{t,n} += lambda_{t,n} Delta_t u_t
 *   du_t = g'_t D + sum_n lambda_{t,n} Delta_t B_{t,n}
 *   dDelta_t = sum_n lambda_{t,n} (B_{t,n} u_t + A[n] abar_{t,n} h_{t-1,n})
 *   dA[n] += lambda_{t,n} Delta_t abar_{t,n} h_{t-1,n}
 *   ddelta_t = dDelta_t * sig(delta_t + Delta_bias);  dDelta_bias += ddelta_t
 *   dD += g'_t u_t
 *
 * All arrays are double, row-major, contiguous.  S6 layouts: u, delta, z, dy
 * [batch, dim, L]; B, C [batch, N, L] (shared across channels); A [dim, N];
 * D, delta_bias [dim]; h0, h_last [batch, dim, N].  SSD layouts: x, z
 * [batch, L, heads, P]; delta [batch, L, heads]; B, C [batch, L, groups, N];
 * A, D, delta_bias [heads]; final_state [batch, heads, P, N].
 * Optional inputs are NULL when absent (D -> 0, z -> no gate, bias -> 0,
 * h0 -> zero state).
 *
 * Every entry point is pinned in tests/test_oracle_pins.py against closed forms,
 * special cases, brute force and finite differences that do not call this file's
 * arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), evaluated without overflow as
 * max(x, 0) + log1p(exp(-|x|)). */
static double softplus_d(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* logistic sigmoid 1 / (1 + e^-x), split by sign so exp never overflows. */
static double sigmoid_d(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* One channel row of the S6 forward.
 * u, delta, z, y: [L] ; A, h0, h_last: [N] ; B, C: [N, L] (this batch's slice).
 * D, bias: scalars for this channel (has_D / has_z select the optional terms).
 * h is caller scratch of N doubles. */
void oracle_s6_fwd_row(int64_t L, int64_t N,
                       const double* u, const double* delta, const double* A,
                       const double* B, const double* C,
                       double D, const double* z, double bias,
                       const double* h0, double* y, double* h_last, double* h) {
    for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double dt = softplus_d(delta[t] + bias);
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double abar = exp(dt * A[n]);
            h[n] = abar * h[n] + dt * B[n * L + t] * u[t];
            acc += C[n * L + t] * h[n];
        }
        acc += D * u[t];
        if (z) acc *= z[t] * sigmoid_d(z[t]);
        y[t] = acc;
    }
    if (h_last)
        for (int64_t n = 0; n < N; ++n) h_last[n] = h[n];
}

/* Full S6 forward over every (batch, channel) row, rows spread over threads. */
int oracle_s6_fwd(int64_t batch, int64_t dim, int64_t L, int64_t N,
                  const double* u, const double* delta, const double* A,
                  const double* B, const double* C, const double* D,
                  const double* z, const double* delta_bias, const double* h0,
                  double* y, double* h_last) {
    int64_t rows = batch * dim;
    int err = 0;
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!h) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < rows; ++r) {
                int64_t b = r / dim, d = r % dim;
                oracle_s6_fwd_row(L, N, u + r * L, delta + r * L, A + d * N,
                                  B + b * N * L, C + b * N * L,
                                  D ? D[d] : 0.0, z ? z + r * L : NULL,
                                  delta_bias ? delta_bias[d] : 0.0,
                                  h0 ? h0 + r * N : NULL, y + r * L,
                                  h_last ? h_last + r * N : NULL, h);
            }
            free(h);
        }
    }
    return err;
}

/* One channel row of the S6 backward.  Recomputes the forward states of the row
 * (an L x N buffer is fine on the CPU), then runs the reverse adjoint.
 * Per-row outputs: du, ddelta, dz [L]; dA_row [N]; *dD_row, *dbias_row.
 * Contributions to the channel-shared grads are ADDED into dB_acc, dC_acc [N, L].
 * hs: scratch (L + 1) * N doubles; lam: scratch N doubles. */
/* S6 forward with another discretisation of the input term; decay, readout,
 * skip and gate as in oracle_s6_fwd_row.
 *  disc 1, zero-order hold ("Mamba 解密" sec. 3 and sec. 5): with the input held
 *    constant over the step, B-bar = (Delta A)^-1 (exp(Delta A) - 1) Delta B, so the
 *    input term is expm1(Delta A_n) / A_n * B_n u (Delta B_n u when A_n = 0).
 *  disc 2, exponential-trapezoidal ("Mamba 解密" sec. 6.3):
 *    h_t = Abar_t h_{t-1} + 1/2 (Bbar_t x_t + Abar_t Bbar_{t-1} x_{t-1}),
 *    read with Bbar_t x_t = Delta_t B_t u_t (the exponential-Euler input term of
 *    sec. 6.3) and no input term before t = 0.
 * eprev: N doubles of scratch. */
void oracle_s6_fwd_disc_row(int disc, int64_t L, int64_t N,
                            const double* u, const double* delta, const double* A,
                            const double* B, const double* C,
                            double D, const double* z, double bias,
                            const double* h0, double* y, double* h_last, double* h, double* eprev) {
    for (int64_t n = 0; n < N; ++n) {
        h[n] = h0 ? h0[n] : 0.0;
        eprev[n] = 0.0;
    }
    for (int64_t t = 0; t < L; ++t) {
        double dt = softplus_d(delta[t] + bias);
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double abar = exp(dt * A[n]);
            double bu = B[n * L + t] * u[t];
            double in;
            if (disc == 1) {
                in = (A[n] != 0.0 ? expm1(dt * A[n]) / A[n] : dt) * bu;
            } else {
                double e = dt * bu;
                in = 0.5 * (e + abar * eprev[n]);
                eprev[n] = e;
            }
            h[n] = abar * h[n] + in;
            acc += C[n * L + t] * h[n];
        }
        acc += D * u[t];
        if (z) acc *= z[t] * sigmoid_d(z[t]);
        y[t] = acc;
    }
    if (h_last)
        for (int64_t n = 0; n < N; ++n) h_last[n] = h[n];
}

int oracle_s6_fwd_disc(int disc, int64_t batch, int64_t dim, int64_t L, int64_t N,
                       const double* u, const double* delta, const double* A,
                       const double* B, const double* C, const double* D,
                       const double* z, const double* delta_bias, const double* h0,
                       double* y, double* h_last) {
    if (disc != 1 && disc != 2) return 2;
    int64_t rows = batch * dim;
    int err = 0;
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)(2 * (N > 0 ? N : 1)));
        if (!h) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < rows; ++r) {
                int64_t b = r / dim, d = r % dim;
                oracle_s6_fwd_disc_row(disc, L, N, u + r * L, delta + r * L, A + d * N,
                                       B + b * N * L, C + b * N * L,
                                       D ? D[d] : 0.0, z ? z + r * L : NULL,
                                       delta_bias ? delta_bias[d] : 0.0,
                                       h0 ? h0 + r * N : NULL, y + r * L,
                                       h_last ? h_last + r * N : NULL, h, h + N);
            }
            free(h);
        }
    }
    return err;
}

void oracle_s6_bwd_row(int64_t L, int64_t N,
                       const double* u, const double* delta, const double* A,
                       const double* B, const double* C,
                       double D, const double* z, double bias, const double* dy,
                       double* du, double* ddelta, double* dz, double* dA_row,
                       double* dD_row, double* dbias_row,
                       double* dB_acc, double* dC_acc, double* hs, double* lam) {
    /* forward: hs[(t + 1) * N + n] = h_{t,n}; hs[0..N) = h_{-1} = 0 */
    for (int64_t n = 0; n < N; ++n) hs[n] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double dt = softplus_d(delta[t] + bias);
        for (int64_t n = 0; n < N; ++n) {
            double abar = exp(dt * A[n]);
            hs[(t + 1) * N + n] = abar * hs[t * N + n] + dt * B[n * L + t] * u[t];
        }
    }
    for (int64_t n = 0; n < N; ++n) { lam[n] = 0.0; dA_row[n] = 0.0; }
    double dD = 0.0, dbias = 0.0;
    /* reverse: lam holds lambda_{t+1} on entry to step t */
    for (int64_t t = L - 1; t >= 0; --t) {
        double x = delta[t] + bias;
        double dt = softplus_d(x);
        double yp = D * u[t];
        for (int64_t n = 0; n < N; ++n) yp += C[n * L + t] * hs[(t + 1) * N + n];
        double gp, dzt = 0.0;
        if (z) {
            double s = sigmoid_d(z[t]);
            gp = dy[t] * z[t] * s;
            dzt = dy[t] * yp * s * (1.0 + z[t] * (1.0 - s));
        } else {
            gp = dy[t];
        }
        double dut = gp * D, dDelta = 0.0;
        dD += gp * u[t];
        double dt_next = (t + 1 < L) ? softplus_d(delta[t + 1] + bias) : 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double abar_next = (t + 1 < L) ? exp(dt_next * A[n]) : 0.0;
            double l = gp * C[n * L + t] + abar_next * lam[n];
            lam[n] = l;
            double abar = exp(dt * A[n]);
            double hprev = hs[t * N + n];
            dC_acc[n * L + t] += gp * hs[(t + 1) * N + n];
            dB_acc[n * L + t] += l * dt * u[t];
            dut += l * dt * B[n * L + t];
            dDelta += l * (B[n * L + t] * u[t] + A[n] * abar * hprev);
            dA_row[n] += l * dt * abar * hprev;
        }
        du[t] = dut;
        ddelta[t] = dDelta * sigmoid_d(x);
        dbias += ddelta[t];
        if (dz) dz[t] = dzt;
    }
    *dD_row = dD;
    *dbias_row = dbias;
}

/* Full S6 backward.  Grads of the channel-shared and per-channel parameters are
 * summed in a fixed order (per-thread partials, then thread order). */
int oracle_s6_bwd(int64_t batch, int64_t dim, int64_t L, int64_t N,
                  const double* u, const double* delta, const double* A,
                  const double* B, const double* C, const double* D,
                  const double* z, const double* delta_bias, const double* dy,
                  double* du, double* ddelta, double* dA, double* dB, double* dC,
                  double* dD, double* dz, double* ddelta_bias) {
    int64_t rows = batch * dim;
    int nth = oracle_num_threads();
    size_t bnl = (size_t)(batch * N * L);
    double* part = (double*)calloc((size_t)nth * (2 * bnl + (size_t)(dim * N + 2 * dim)), sizeof(double));
    if (!part) return 1;
    int err = 0;
#pragma omp parallel num_threads(nth)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double* pB = part + (size_t)tid * (2 * bnl + (size_t)(dim * N + 2 * dim));
        double* pC = pB + bnl;
        double* pA = pC + bnl;
        double* pD = pA + dim * N;
        double* pbias = pD + dim;
        double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N + N + 1));
        double* dArow = (double*)malloc(sizeof(double) * (size_t)(N + 1));
        if (!hs || !dArow) {
#pragma omp atomic write
            err = 1;
        } else {
            double* lam = hs + (L + 1) * N;
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                int64_t b = r / dim, d = r % dim;
                double dDr, dbr;
                oracle_s6_bwd_row(L, N, u + r * L, delta + r * L, A + d * N,
                                  B + b * N * L, C + b * N * L, D ? D[d] : 0.0,
                                  z ? z + r * L : NULL,
                                  delta_bias ? delta_bias[d] : 0.0, dy + r * L,
                                  du + r * L, ddelta + r * L, z ? dz + r * L : NULL,
                                  dArow, &dDr, &dbr, pB + b * N * L, pC + b * N * L,
                                  hs, lam);
                for (int64_t n = 0; n < N; ++n) pA[d * N + n] += dArow[n];
                pD[d] += dDr;
                pbias[d] += dbr;
            }
        }
        free(hs);
        free(dArow);
    }
    if (!err) {
        memset(dB, 0, sizeof(double) * bnl);
        memset(dC, 0, sizeof(double) * bnl);
        memset(dA, 0, sizeof(double) * (size_t)(dim * N));
        double* tD = (double*)calloc((size_t)(2 * dim), sizeof(double));
        if (!tD) { free(part); return 1; }
        for (int t = 0; t < nth; ++t) {
            double* pB = part + (size_t)t * (2 * bnl + (size_t)(dim * N + 2 * dim));
            double* pC = pB + bnl;
            double* pA = pC + bnl;
            double* pD = pA + dim * N;
            double* pbias = pD + dim;
            for (size_t i = 0; i < bnl; ++i) { dB[i] += pB[i]; dC[i] += pC[i]; }
            for (int64_t i = 0; i < dim * N; ++i) dA[i] += pA[i];
            for (int64_t i = 0; i < dim; ++i) { tD[i] += pD[i]; tD[dim + i] += pbias[i]; }
        }
        if (dD) memcpy(dD, tD, sizeof(double) * (size_t)dim);
        if (ddelta_bias) memcpy(ddelta_bias, tD + dim, sizeof(double) * (size_t)dim);
        free(tD);
    }
    free(part);
    return err;
}

/* One (batch, head) of the SSD forward: the scalar-A recurrence on a P x N state.
 * x, z, y: strided rows, element (t, p) at [t * sx + p]; delta: [t * sd];
 * B, C: element (t, n) at [t * sb + n].  H: P x N scratch (and final state out). */
void oracle_ssd_fwd_head(int64_t L, int64_t P, int64_t N,
                         const double* x, int64_t sx, const double* delta, int64_t sd,
                         double A, const double* B, const double* C, int64_t sb,
                         double D, const double* z, double bias,
                         double* y, double* H) {
    for (int64_t i = 0; i < P * N; ++i) H[i] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double dt = softplus_d(delta[t * sd] + bias);
        double a = exp(dt * A);
        for (int64_t p = 0; p < P; ++p) {
            double xp = x[t * sx + p];
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double hv = a * H[p * N + n] + dt * xp * B[t * sb + n];
                H[p * N + n] = hv;
                acc += hv * C[t * sb + n];
            }
            acc += D * xp;
            if (z) {
                double zv = z[t * sx + p];
                acc *= zv * sigmoid_d(zv);
            }
            y[t * sx + p] = acc;
        }
    }
}

/* Full SSD forward over every (batch, head). */
int oracle_ssd_fwd(int64_t batch, int64_t L, int64_t nheads, int64_t P, int64_t N,
                   int64_t ngroups, const double* x, const double* delta,
                   const double* A, const double* B, const double* C,
                   const double* D, const double* z, const double* delta_bias,
                   double* y, double* final_state) {
    if (ngroups <= 0 || nheads % ngroups != 0) return 2;
    int64_t hpg = nheads / ngroups;
    int err = 0;
#pragma omp parallel
    {
        double* H = (double*)malloc(sizeof(double) * (size_t)(P * N > 0 ? P * N : 1));
        if (!H) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < batch * nheads; ++bh) {
                int64_t b = bh / nheads, h = bh % nheads, g = h / hpg;
                const double* xb = x + (b * L * nheads + h) * P;
                oracle_ssd_fwd_head(L, P, N, xb, nheads * P,
                                    delta + b * L * nheads + h, nheads, A[h],
                                    B + (b * L * ngroups + g) * N,
                                    C + (b * L * ngroups + g) * N, ngroups * N,
                                    D ? D[h] : 0.0,
                                    z ? z + (b * L * nheads + h) * P : NULL,
                                    delta_bias ? delta_bias[h] : 0.0,
                                    y + (b * L * nheads + h) * P, H);
                if (final_state)
                    memcpy(final_state + bh * P * N, H, sizeof(double) * (size_t)(P * N));
            }
            free(H);
        }
    }
    return err;
}
