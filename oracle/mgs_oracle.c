/*
 * Float64 CPU oracle for the three scan primitives of the minGRU family.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Every function is the plain definition of the recurrence, written out as a
 * sequential loop over t in double precision, one independent lane at a time
 * (OpenMP only splits the lanes across host threads; the arithmetic inside a
 * lane is the textbook order).
 *
 * Sources.  The operations are the scan primitives named on the mingru-scans
 * pages ("mingru-scans" home page, scan-op speedup table: matrix_scan,
 * matrix_affine_scan, parallel_scan_log; "Run the benchmarks", Step 2 timing
 * matrix).  The pages name them but print no formula, so each recurrence below
 * is the standard one for its name:
 *   matrix_affine_scan  h_t = A_t h_{t-1} + b_t            (k x k blocks)
 *   matrix_scan         P_t = A_t P_{t-1},  P_0 = I
 *   parallel_scan_log   h_t = e^{lc_t} h_{t-1} + e^{lv_t}  in log space,
 *                       Heinsen (2023, arXiv:2311.06281), cited on the
 *                       home page's lineage paragraph.
 *   Givens affine scan  matrix_affine_scan with A_t = G(theta_t) diag(a_t),
 *   Givens matrix scan  matrix_scan with A_t = G(theta_t): the brick-wall
 *                       rotation mesh of GivensMinGRU, fed by its angles.
 *   delta rule          S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,
 *                       o_t = S_t q_t (DeltaNet, behind DeltaMinGRU).
 * Backward passes are the adjoint (reverse-mode) recurrences of those maps.
 *
 * Layouts (row-major, contiguous, double):
 *   A  [B][T][H][K][K]   A[...][i][j] multiplies h[j] into output row i
 *   b, h, grad_h, db  [B][T][H][K];  h0, dh0  [B][H][K]
 *   P, grad_P, dA  [B][T][H][K][K]
 *   lc, lv, h, log_h, grad_h, d_lc, d_lv  [B][T][D];  log_h0, d_log_h0 [B][D]
 * Output index t runs over 1..T and is stored at position t-1; the initial
 * state (h_0 / P_0) is not part of the output.
 *
 * Parity status: every function here is pinned by the CPU tests (closed
 * forms, invariants, brute force, finite differences, adjoint identities).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* matrix_affine_scan                                                   */
/* ------------------------------------------------------------------ */

/* Forward: h_t = A_t h_{t-1} + b_t for t = 1..T, h_0 = h0 (zeros if h0 is
 * NULL), independently for every (batch, head) lane. */
void oracle_mas_fwd(const double *A, const double *bv, const double *h0,
                    double *h, int64_t B, int64_t T, int64_t H, int64_t K)
{
    int64_t lanes = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *prev = (double *)malloc(sizeof(double) * (size_t)K);
        for (int64_t i = 0; i < K; ++i)
            prev[i] = h0 ? h0[(bb * H + hd) * K + i] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double *At = A + (((bb * T + t) * H + hd) * K) * K;
            const double *bt = bv + ((bb * T + t) * H + hd) * K;
            double *ht = h + ((bb * T + t) * H + hd) * K;
            for (int64_t i = 0; i < K; ++i) {
                double s = bt[i];
                for (int64_t j = 0; j < K; ++j)
                    s += At[i * K + j] * prev[j];
                ht[i] = s;
            }
            for (int64_t i = 0; i < K; ++i)
                prev[i] = ht[i];
        }
        free(prev);
    }
}

/* Backward of the forward above for the loss L = sum_t <grad_h_t, h_t>.
 * The forward states are recomputed here from (A, b, h0), so nothing from any
 * other implementation enters.  With lambda_t = dL/dh_t (total derivative):
 *   lambda_T = g_T,  lambda_t = g_t + A_{t+1}^T lambda_{t+1},
 *   dL/db_t = lambda_t,  dL/dA_t = lambda_t h_{t-1}^T,
 *   dL/dh_0 = A_1^T lambda_1.
 * dh0 may be NULL (not written). */
void oracle_mas_bwd(const double *A, const double *bv, const double *h0,
                    const double *gh, double *dA, double *db, double *dh0,
                    int64_t B, int64_t T, int64_t H, int64_t K)
{
    int64_t lanes = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        /* states[t] holds h_t for t = 0..T */
        double *states = (double *)malloc(sizeof(double) * (size_t)((T + 1) * K));
        double *lam = (double *)malloc(sizeof(double) * (size_t)K);
        double *nxt = (double *)malloc(sizeof(double) * (size_t)K);
        for (int64_t i = 0; i < K; ++i)
            states[i] = h0 ? h0[(bb * H + hd) * K + i] : 0.0;
        for (int64_t t = 1; t <= T; ++t) {
            const double *At = A + (((bb * T + (t - 1)) * H + hd) * K) * K;
            const double *bt = bv + ((bb * T + (t - 1)) * H + hd) * K;
            for (int64_t i = 0; i < K; ++i) {
                double s = bt[i];
                for (int64_t j = 0; j < K; ++j)
                    s += At[i * K + j] * states[(t - 1) * K + j];
                states[t * K + i] = s;
            }
        }
        /* reverse sweep; nxt = A_{t+1}^T lambda_{t+1} (zero at t = T) */
        for (int64_t i = 0; i < K; ++i)
            nxt[i] = 0.0;
        for (int64_t t = T; t >= 1; --t) {
            const double *gt = gh + ((bb * T + (t - 1)) * H + hd) * K;
            const double *At = A + (((bb * T + (t - 1)) * H + hd) * K) * K;
            double *dAt = dA + (((bb * T + (t - 1)) * H + hd) * K) * K;
            double *dbt = db + ((bb * T + (t - 1)) * H + hd) * K;
            for (int64_t i = 0; i < K; ++i)
                lam[i] = gt[i] + nxt[i];
            for (int64_t i = 0; i < K; ++i) {
                dbt[i] = lam[i];
                for (int64_t j = 0; j < K; ++j)
                    dAt[i * K + j] = lam[i] * states[(t - 1) * K + j];
            }
            for (int64_t j = 0; j < K; ++j) {
                double s = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    s += At[i * K + j] * lam[i];
                nxt[j] = s;
            }
        }
        if (dh0)
            for (int64_t j = 0; j < K; ++j)
                dh0[(bb * H + hd) * K + j] = T > 0 ? nxt[j] : 0.0;
        free(states);
        free(lam);
        free(nxt);
    }
}

/* ------------------------------------------------------------------ */
/* matrix_scan                                                          */
/* ------------------------------------------------------------------ */

/* Forward: prefix products P_t = A_t P_{t-1}, P_0 = I, per lane. */
void oracle_ms_fwd(const double *A, double *P, int64_t B, int64_t T,
                   int64_t H, int64_t K)
{
    int64_t lanes = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *prev = (double *)malloc(sizeof(double) * (size_t)(K * K));
        for (int64_t i = 0; i < K; ++i)
            for (int64_t j = 0; j < K; ++j)
                prev[i * K + j] = (i == j) ? 1.0 : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double *At = A + (((bb * T + t) * H + hd) * K) * K;
            double *Pt = P + (((bb * T + t) * H + hd) * K) * K;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t m = 0; m < K; ++m)
                        s += At[i * K + m] * prev[m * K + j];
                    Pt[i * K + j] = s;
                }
            memcpy(prev, Pt, sizeof(double) * (size_t)(K * K));
        }
        free(prev);
    }
}

/* Backward for L = sum_t <G_t, P_t>_F with Lambda_t = dL/dP_t (total):
 *   Lambda_T = G_T,  Lambda_t = G_t + A_{t+1}^T Lambda_{t+1},
 *   dL/dA_t = Lambda_t P_{t-1}^T  with P_0 = I.
 * Prefix products are recomputed here from A. */
void oracle_ms_bwd(const double *A, const double *gP, double *dA, int64_t B,
                   int64_t T, int64_t H, int64_t K)
{
    int64_t lanes = B * H;
    int64_t KK = K * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *prods = (double *)malloc(sizeof(double) * (size_t)((T + 1) * KK));
        double *lam = (double *)malloc(sizeof(double) * (size_t)KK);
        double *nxt = (double *)malloc(sizeof(double) * (size_t)KK);
        for (int64_t i = 0; i < K; ++i)
            for (int64_t j = 0; j < K; ++j)
                prods[i * K + j] = (i == j) ? 1.0 : 0.0;
        for (int64_t t = 1; t <= T; ++t) {
            const double *At = A + (((bb * T + (t - 1)) * H + hd) * K) * K;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t m = 0; m < K; ++m)
                        s += At[i * K + m] * prods[(t - 1) * KK + m * K + j];
                    prods[t * KK + i * K + j] = s;
                }
        }
        for (int64_t e = 0; e < KK; ++e)
            nxt[e] = 0.0;
        for (int64_t t = T; t >= 1; --t) {
            const double *Gt = gP + (((bb * T + (t - 1)) * H + hd) * K) * K;
            const double *At = A + (((bb * T + (t - 1)) * H + hd) * K) * K;
            double *dAt = dA + (((bb * T + (t - 1)) * H + hd) * K) * K;
            const double *Pprev = prods + (t - 1) * KK;
            for (int64_t e = 0; e < KK; ++e)
                lam[e] = Gt[e] + nxt[e];
            /* dA_t[i][m] = sum_j Lambda_t[i][j] * P_{t-1}[m][j] */
            for (int64_t i = 0; i < K; ++i)
                for (int64_t m = 0; m < K; ++m) {
                    double s = 0.0;
                    for (int64_t j = 0; j < K; ++j)
                        s += lam[i * K + j] * Pprev[m * K + j];
                    dAt[i * K + m] = s;
                }
            /* nxt = A_t^T Lambda_t: nxt[m][j] = sum_i A_t[i][m] Lambda_t[i][j] */
            for (int64_t m = 0; m < K; ++m)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t i = 0; i < K; ++i)
                        s += At[i * K + m] * lam[i * K + j];
                    nxt[m * K + j] = s;
                }
        }
        free(prods);
        free(lam);
        free(nxt);
    }
}

/* ------------------------------------------------------------------ */
/* parallel_scan_log                                                    */
/* ------------------------------------------------------------------ */

/* log(e^x + e^y) with -inf handled exactly; max-shifted so nothing
 * overflows. */
static double logaddexp_d(double x, double y)
{
    double m = x > y ? x : y;
    if (m == -INFINITY)
        return -INFINITY;
    return m + log1p(exp(-fabs(x - y)));
}

/* Forward of the diagonal log-space scan, per (batch, channel) lane:
 *   log h_t = log(e^{lc_t + log h_{t-1}} + e^{lv_t}),  log h_0 = log_h0
 * (or -inf, i.e. h_0 = 0, when log_h0 is NULL); h_t = exp(log h_t).
 * This is the recurrence h_t = a_t h_{t-1} + v_t with a = e^lc, v = e^lv,
 * whose closed form is Heinsen's exp(a*_t + logcumsumexp(lv - a*)).
 * log_h may be NULL. */
void oracle_psl_fwd(const double *lc, const double *lv, const double *log_h0,
                    double *h, double *log_h, int64_t B, int64_t T, int64_t D)
{
    int64_t lanes = B * D;
#pragma omp parallel for schedule(static)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / D, d = lane % D;
        double L = log_h0 ? log_h0[bb * D + d] : -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            int64_t idx = (bb * T + t) * D + d;
            L = logaddexp_d(lc[idx] + L, lv[idx]);
            h[idx] = exp(L);
            if (log_h)
                log_h[idx] = L;
        }
    }
}

/* Backward for L = sum_t grad_h_t * h_t, per lane, with lambda_t = dL/dh_t:
 *   lambda_T = g_T,  lambda_t = g_t + a_{t+1} lambda_{t+1},  a_t = e^{lc_t},
 *   dL/dlv_t = lambda_t e^{lv_t},
 *   dL/dlc_t = lambda_t a_t h_{t-1},
 *   dL/dlog_h0 = lambda_1 a_1 h_0    (written only when log_h0 is given).
 * The forward states are recomputed here (in log space, as above). */
void oracle_psl_bwd(const double *lc, const double *lv, const double *log_h0,
                    const double *gh, double *dlc, double *dlv,
                    double *dlog_h0, int64_t B, int64_t T, int64_t D)
{
    int64_t lanes = B * D;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / D, d = lane % D;
        /* hs[t] = h_t for t = 0..T */
        double *hs = (double *)malloc(sizeof(double) * (size_t)(T + 1));
        double L = log_h0 ? log_h0[bb * D + d] : -INFINITY;
        hs[0] = exp(L);
        for (int64_t t = 1; t <= T; ++t) {
            int64_t idx = (bb * T + (t - 1)) * D + d;
            L = logaddexp_d(lc[idx] + L, lv[idx]);
            hs[t] = exp(L);
        }
        double nxt = 0.0; /* a_{t+1} lambda_{t+1}, zero at t = T */
        double lam = 0.0;
        for (int64_t t = T; t >= 1; --t) {
            int64_t idx = (bb * T + (t - 1)) * D + d;
            double a = exp(lc[idx]);
            lam = gh[idx] + nxt;
            dlv[idx] = lam * exp(lv[idx]);
            dlc[idx] = lam * a * hs[t - 1];
            nxt = a * lam;
        }
        if (dlog_h0)
            dlog_h0[bb * D + d] = T > 0 ? nxt * hs[0] : 0.0;
        free(hs);
    }
}

/* ------------------------------------------------------------------ */
/* linear_scan                                                          */
/* ------------------------------------------------------------------ */

/* Forward of the diagonal linear recurrence, per (batch, channel) lane:
 *   h_t = a_t h_{t-1} + b_t,  h_0 = h0 (zeros when NULL).
 * Signed coefficients are allowed.  Layout [B][T][D], h0 [B][D]. */
void oracle_linear_fwd(const double *a, const double *bv, const double *h0, double *h,
                       int64_t B, int64_t T, int64_t D)
{
    int64_t lanes = B * D;
#pragma omp parallel for schedule(static)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / D, d = lane % D;
        double x = h0 ? h0[bb * D + d] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t idx = (bb * T + t) * D + d;
            x = a[idx] * x + bv[idx];
            h[idx] = x;
        }
    }
}

/* Backward for L = sum_t g_t h_t:  lambda_T = g_T,
 * lambda_t = g_t + a_{t+1} lambda_{t+1};  db_t = lambda_t;
 * da_t = lambda_t h_{t-1};  dh0 = a_1 lambda_1 (dh0 may be NULL).
 * The forward states are recomputed from (a, b, h0). */
void oracle_linear_bwd(const double *a, const double *bv, const double *h0, const double *gh,
                       double *da, double *db, double *dh0, int64_t B, int64_t T, int64_t D)
{
    int64_t lanes = B * D;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / D, d = lane % D;
        double *hs = (double *)malloc(sizeof(double) * (size_t)(T + 1));
        hs[0] = h0 ? h0[bb * D + d] : 0.0;
        for (int64_t t = 1; t <= T; ++t) {
            int64_t idx = (bb * T + (t - 1)) * D + d;
            hs[t] = a[idx] * hs[t - 1] + bv[idx];
        }
        double nxt = 0.0; /* a_{t+1} lambda_{t+1} */
        for (int64_t t = T; t >= 1; --t) {
            int64_t idx = (bb * T + (t - 1)) * D + d;
            double lam = gh[idx] + nxt;
            db[idx] = lam;
            da[idx] = lam * hs[t - 1];
            nxt = a[idx] * lam;
        }
        if (dh0)
            dh0[bb * D + d] = nxt;
        free(hs);
    }
}

/* ------------------------------------------------------------------ */
/* Givens-mesh (angle-parameterised) matrix_affine_scan / matrix_scan   */
/* ------------------------------------------------------------------ */

/* The GivensMinGRU transition ("mingru-scans" home page, lineage paragraph:
 * the brick-wall mesh of Clements et al. 2016 / EUNN, built from Golub & Van
 * Loan's plane rotations; "Run the benchmarks", Step 3: the angle-fused
 * backward).  For K coordinates the mesh has K layers; layer l = 1..K rotates
 * the disjoint pairs (p, p+1) with p = 0, 2, 4, ... for odd l and p = 1, 3,
 * 5, ... for even l (p+1 < K, no wrap-around), K(K-1)/2 angles in all,
 * consumed layer by layer, pairs ascending.  The rotation of angle th on pair
 * (p, p+1) maps (x_p, x_{p+1}) to (cos th x_p - sin th x_{p+1},
 * sin th x_p + cos th x_{p+1}).  G(theta) = L_K ... L_1 (layer 1 first).
 *
 * givens_matrix builds M = G(theta) diag(a) (diag(a) = I when a is NULL) by
 * left-multiplying the layers onto diag(a) one rotation at a time.  When
 * deriv >= 0, the rotation of angle `deriv` is replaced by its derivative
 * with respect to that angle, [[-sin, -cos], [cos, -sin]] on its pair and zero
 * on every other row, so M becomes dM/dtheta_deriv. */
static void givens_matrix(const double *th, const double *a, int64_t K, int64_t deriv, double *M)
{
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < K; ++j)
            M[i * K + j] = (i == j) ? (a ? a[j] : 1.0) : 0.0;
    int64_t idx = 0;
    for (int64_t l = 1; l <= K; ++l) {
        for (int64_t p = (l % 2 == 1) ? 0 : 1; p + 1 < K; p += 2, ++idx) {
            double c = cos(th[idx]), s = sin(th[idx]);
            if (idx == deriv) {
                for (int64_t col = 0; col < K; ++col) {
                    double x = M[p * K + col], y = M[(p + 1) * K + col];
                    for (int64_t r = 0; r < K; ++r)
                        if (r != p && r != p + 1)
                            M[r * K + col] = 0.0;
                    M[p * K + col] = -s * x - c * y;
                    M[(p + 1) * K + col] = c * x - s * y;
                }
            } else {
                for (int64_t col = 0; col < K; ++col) {
                    double x = M[p * K + col], y = M[(p + 1) * K + col];
                    M[p * K + col] = c * x - s * y;
                    M[(p + 1) * K + col] = s * x + c * y;
                }
            }
        }
    }
}

/* Forward of the Givens affine scan, per (batch, head) lane:
 *   h_t = G(theta_t) diag(a_t) h_{t-1} + b_t,  h_0 = h0 (zeros when NULL),
 * i.e. matrix_affine_scan with A_t = G(theta_t) diag(a_t) (a NULL: A_t =
 * G(theta_t)).  Layouts: theta [B][T][H][N], N = K(K-1)/2; a, b, h
 * [B][T][H][K]; h0 [B][H][K]. */
void oracle_gas_fwd(const double *theta, const double *a, const double *bv, const double *h0,
                    double *h, int64_t B, int64_t T, int64_t H, int64_t K)
{
    int64_t N = K * (K - 1) / 2, lanes = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *M = (double *)malloc(sizeof(double) * (size_t)(K * K));
        double *prev = (double *)malloc(sizeof(double) * (size_t)K);
        for (int64_t i = 0; i < K; ++i)
            prev[i] = h0 ? h0[(bb * H + hd) * K + i] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t st = (bb * T + t) * H + hd;
            givens_matrix(theta + st * N, a ? a + st * K : NULL, K, -1, M);
            double *ht = h + st * K;
            for (int64_t i = 0; i < K; ++i) {
                double s = bv[st * K + i];
                for (int64_t j = 0; j < K; ++j)
                    s += M[i * K + j] * prev[j];
                ht[i] = s;
            }
            memcpy(prev, ht, sizeof(double) * (size_t)K);
        }
        free(M);
        free(prev);
    }
}

/* Backward of the Givens affine scan for L = sum_t <g_t, h_t>, by the chain
 * rule through A_t = G(theta_t) diag(a_t):
 *   lambda_T = g_T,  lambda_t = g_t + A_{t+1}^T lambda_{t+1},  db_t = lambda_t,
 *   dA_t = lambda_t h_{t-1}^T,
 *   dtheta_t[n] = <dA_t, dA_t/dtheta_n>_F,  da_t[j] = sum_r dA_t[r][j] G_t[r][j],
 *   dh0 = A_1^T lambda_1.
 * The states h_t are recomputed from the inputs.  a, da may be NULL (then
 * A_t = G(theta_t) and da is not produced); dh0 may be NULL. */
void oracle_gas_bwd(const double *theta, const double *a, const double *bv, const double *h0,
                    const double *gh, double *dtheta, double *da, double *db, double *dh0,
                    int64_t B, int64_t T, int64_t H, int64_t K)
{
    int64_t N = K * (K - 1) / 2, lanes = B * H, KK = K * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *states = (double *)malloc(sizeof(double) * (size_t)((T + 1) * K));
        double *M = (double *)malloc(sizeof(double) * (size_t)KK);
        double *dM = (double *)malloc(sizeof(double) * (size_t)KK);
        double *dAt = (double *)malloc(sizeof(double) * (size_t)KK);
        double *lam = (double *)malloc(sizeof(double) * (size_t)K);
        double *nxt = (double *)malloc(sizeof(double) * (size_t)K);
        for (int64_t i = 0; i < K; ++i)
            states[i] = h0 ? h0[(bb * H + hd) * K + i] : 0.0;
        for (int64_t t = 1; t <= T; ++t) {
            int64_t st = (bb * T + (t - 1)) * H + hd;
            givens_matrix(theta + st * N, a ? a + st * K : NULL, K, -1, M);
            for (int64_t i = 0; i < K; ++i) {
                double s = bv[st * K + i];
                for (int64_t j = 0; j < K; ++j)
                    s += M[i * K + j] * states[(t - 1) * K + j];
                states[t * K + i] = s;
            }
        }
        for (int64_t i = 0; i < K; ++i)
            nxt[i] = 0.0;
        for (int64_t t = T; t >= 1; --t) {
            int64_t st = (bb * T + (t - 1)) * H + hd;
            const double *th = theta + st * N;
            const double *at = a ? a + st * K : NULL;
            for (int64_t i = 0; i < K; ++i) {
                lam[i] = gh[st * K + i] + nxt[i];
                db[st * K + i] = lam[i];
            }
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j)
                    dAt[i * K + j] = lam[i] * states[(t - 1) * K + j];
            for (int64_t n = 0; n < N; ++n) {
                givens_matrix(th, at, K, n, dM);
                double s = 0.0;
                for (int64_t e = 0; e < KK; ++e)
                    s += dAt[e] * dM[e];
                dtheta[st * N + n] = s;
            }
            if (da) {
                givens_matrix(th, NULL, K, -1, M);
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t r = 0; r < K; ++r)
                        s += dAt[r * K + j] * M[r * K + j];
                    da[st * K + j] = s;
                }
            }
            givens_matrix(th, at, K, -1, M);
            for (int64_t j = 0; j < K; ++j) {
                double s = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    s += M[i * K + j] * lam[i];
                nxt[j] = s;
            }
        }
        if (dh0)
            for (int64_t i = 0; i < K; ++i)
                dh0[(bb * H + hd) * K + i] = nxt[i];
        free(states);
        free(M);
        free(dM);
        free(dAt);
        free(lam);
        free(nxt);
    }
}

/* Forward of the Givens matrix scan: P_t = G(theta_t) P_{t-1}, P_0 = I.
 * theta [B][T][H][N] -> P [B][T][H][K][K]. */
void oracle_gms_fwd(const double *theta, double *P, int64_t B, int64_t T, int64_t H, int64_t K)
{
    int64_t N = K * (K - 1) / 2, lanes = B * H, KK = K * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *M = (double *)malloc(sizeof(double) * (size_t)KK);
        double *prev = (double *)malloc(sizeof(double) * (size_t)KK);
        for (int64_t i = 0; i < K; ++i)
            for (int64_t j = 0; j < K; ++j)
                prev[i * K + j] = (i == j) ? 1.0 : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t st = (bb * T + t) * H + hd;
            givens_matrix(theta + st * N, NULL, K, -1, M);
            double *Pt = P + st * KK;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t m = 0; m < K; ++m)
                        s += M[i * K + m] * prev[m * K + j];
                    Pt[i * K + j] = s;
                }
            memcpy(prev, Pt, sizeof(double) * (size_t)KK);
        }
        free(M);
        free(prev);
    }
}

/* Backward of the Givens matrix scan for L = sum_t <G_t, P_t>_F:
 *   Lambda_T = G_T,  Lambda_t = G_t + A_{t+1}^T Lambda_{t+1},  A_t = G(theta_t),
 *   dA_t = Lambda_t P_{t-1}^T (P_0 = I),  dtheta_t[n] = <dA_t, dA_t/dtheta_n>_F.
 * gP [B][T][H][K][K] -> dtheta [B][T][H][N]; prefix products recomputed. */
void oracle_gms_bwd(const double *theta, const double *gP, double *dtheta, int64_t B, int64_t T,
                    int64_t H, int64_t K)
{
    int64_t N = K * (K - 1) / 2, lanes = B * H, KK = K * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *prods = (double *)malloc(sizeof(double) * (size_t)((T + 1) * KK));
        double *M = (double *)malloc(sizeof(double) * (size_t)KK);
        double *dM = (double *)malloc(sizeof(double) * (size_t)KK);
        double *dAt = (double *)malloc(sizeof(double) * (size_t)KK);
        double *lam = (double *)malloc(sizeof(double) * (size_t)KK);
        double *nxt = (double *)malloc(sizeof(double) * (size_t)KK);
        for (int64_t i = 0; i < K; ++i)
            for (int64_t j = 0; j < K; ++j)
                prods[i * K + j] = (i == j) ? 1.0 : 0.0;
        for (int64_t t = 1; t <= T; ++t) {
            int64_t st = (bb * T + (t - 1)) * H + hd;
            givens_matrix(theta + st * N, NULL, K, -1, M);
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t m = 0; m < K; ++m)
                        s += M[i * K + m] * prods[(t - 1) * KK + m * K + j];
                    prods[t * KK + i * K + j] = s;
                }
        }
        for (int64_t e = 0; e < KK; ++e)
            nxt[e] = 0.0;
        for (int64_t t = T; t >= 1; --t) {
            int64_t st = (bb * T + (t - 1)) * H + hd;
            const double *th = theta + st * N;
            const double *Pprev = prods + (t - 1) * KK;
            for (int64_t e = 0; e < KK; ++e)
                lam[e] = gP[st * KK + e] + nxt[e];
            for (int64_t i = 0; i < K; ++i)
                for (int64_t m = 0; m < K; ++m) {
                    double s = 0.0;
                    for (int64_t j = 0; j < K; ++j)
                        s += lam[i * K + j] * Pprev[m * K + j];
                    dAt[i * K + m] = s;
                }
            for (int64_t n = 0; n < N; ++n) {
                givens_matrix(th, NULL, K, n, dM);
                double s = 0.0;
                for (int64_t e = 0; e < KK; ++e)
                    s += dAt[e] * dM[e];
                dtheta[st * N + n] = s;
            }
            givens_matrix(th, NULL, K, -1, M);
            for (int64_t m = 0; m < K; ++m)
                for (int64_t j = 0; j < K; ++j) {
                    double s = 0.0;
                    for (int64_t i = 0; i < K; ++i)
                        s += M[i * K + m] * lam[i * K + j];
                    nxt[m * K + j] = s;
                }
        }
        free(prods);
        free(M);
        free(dM);
        free(dAt);
        free(lam);
        free(nxt);
    }
}

/* ------------------------------------------------------------------ */
/* delta rule (DeltaNet), forward                                       */
/* ------------------------------------------------------------------ */

/* DeltaMinGRU's recurrence ("mingru-scans" home page, lineage paragraph:
 * DeltaMinGRU reimplements DeltaNet, Yang et al. 2024, arXiv:2406.06484,
 * whose chunked WY form is its parallel forward).  The delta rule, per
 * (batch, head) lane, with a d_v x d_k state S (here d_v = d_k = D):
 *   S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,   o_t = S_t q_t,
 * S_0 = S0 (zeros when NULL).  Layouts: q, k, v, o [B][T][H][D];
 * beta [B][T][H]; S0, S_T [B][H][D][D] with S[i][j], i the value index.
 * S_T (the state after step T) is written when not NULL. */
void oracle_delta_fwd(const double *q, const double *k, const double *v, const double *beta,
                      const double *S0, double *o, double *ST, int64_t B, int64_t T, int64_t H,
                      int64_t D)
{
    int64_t lanes = B * H, DD = D * D;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lane = 0; lane < lanes; ++lane) {
        int64_t bb = lane / H, hd = lane % H;
        double *S = (double *)malloc(sizeof(double) * (size_t)DD);
        double *Sk = (double *)malloc(sizeof(double) * (size_t)D);
        for (int64_t e = 0; e < DD; ++e)
            S[e] = S0 ? S0[(bb * H + hd) * DD + e] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t st = (bb * T + t) * H + hd;
            const double *kt = k + st * D, *vt = v + st * D, *qt = q + st * D;
            double bt = beta[st];
            for (int64_t i = 0; i < D; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < D; ++j)
                    s += S[i * D + j] * kt[j];
                Sk[i] = s;
            }
            for (int64_t i = 0; i < D; ++i)
                for (int64_t j = 0; j < D; ++j)
                    S[i * D + j] += bt * (vt[i] - Sk[i]) * kt[j];
            for (int64_t i = 0; i < D; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < D; ++j)
                    s += S[i * D + j] * qt[j];
                o[st * D + i] = s;
            }
        }
        if (ST)
            memcpy(ST + (bb * H + hd) * DD, S, sizeof(double) * (size_t)DD);
        free(S);
        free(Sk);
    }
}

/* Number of host threads the OpenMP loops above use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
