/*
 * sdtw_oracle.c -- plain fp64 CPU oracle for batched Soft-DTW.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct statement
 * of what the CUDA library computes. Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What is computed (all in double precision, from the caller's inputs):
 *
 *  Cost.  C[i,j] = sum_k (x[i,k] - y[j,k])^2, squared Euclidean distance with
 *         no 1/2 factor (SoftDTW-CUDA (PyTorch + Numba) README, "Notes":
 *         squared Euclidean distances are always >= 0; "Fused Mode":
 *         dist="sqeuclidean").
 *
 *  Forward.  Soft-DTW of Cuturi & Blondel (ICML 2017), the method the README's
 *         "Acknowledgments" names:
 *           R[0,0] = 0,  R[i,0] = R[0,j] = +inf  (i,j >= 1),
 *           R[i,j] = C[i,j] + softmin_g(R[i-1,j-1], R[i-1,j], R[i,j-1]),
 *           softmin_g(a) = -g log sum exp(-a/g),
 *         evaluated with the minimum as shift; infinite predecessors are left
 *         out of the sum. The value is R[N,M] and can be negative
 *         (README, "Notes").
 *
 *  Backward (log space).  The alignment matrix E = dR[N,M]/dC is obtained from
 *         the reverse recursion done with log-sum-exp, and exp is applied only
 *         after the backward DP (SoftDTW-CUDA-Torch paper, abstract,
 *         contribution (2); review page, "proposed method", second bullet):
 *           logE[N,M] = 0,
 *           logE[i,j] = LSE over successors s in {(i+1,j),(i,j+1),(i+1,j+1)}
 *                       that lie inside the matrix of
 *                       logE[s] + (R[s] - C[s] - R[i,j]) / g,
 *           E = exp(logE).
 *         Successors outside the matrix are omitted (no inf - inf).
 *
 *  Gradients (chain rule through C):
 *           grad_x[i,k] = g_b * 2 sum_j E[i,j] (x[i,k] - y[j,k]),
 *           grad_y[j,k] = g_b * 2 sum_i E[i,j] (y[j,k] - x[i,k]),
 *         with g_b the upstream derivative of the b-th loss.
 *
 *  Normalized (README, "Normalization"):
 *           s(x,y) - (s(x,x) + s(y,y)) / 2,  equal shapes only.
 *         s(x,x) takes x in both slots, so its x-derivative is gx + gy.
 *
 *  Barycenter step (README, "Time Series Barycenters (Averaging)"; review
 *         page, "proposed method", fifth bullet: Adam on the Soft-DTW
 *         objective): L(z) = (1/K) sum_k s(z, X_k); Adam of Kingma & Ba with
 *         bias correction, step t (1-based):
 *           m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 *           z <- z - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps).
 *         Parity of the full barycenter loop is pinned only through this
 *         step (no page prints a barycenter trajectory).
 *
 * Layout: row-major, x (B,N,D), y (B,M,D), grads like their inputs.
 * Errors: functions return 0 on success, -1 on a bad argument or a failed
 * allocation.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- single problem ------------------------------------------------------ */

/* C (N,M) from x (N,D) and y (M,D). */
void oracle_sqeuclid(const double* x, const double* y, int N, int M, int D, double* C)
{
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < M; ++j) {
            double acc = 0.0;
            for (int k = 0; k < D; ++k) {
                double d = x[(size_t)i * D + k] - y[(size_t)j * D + k];
                acc += d * d;
            }
            C[(size_t)i * M + j] = acc;
        }
}

/* R ((N+1),(M+1)) with borders; returns R[N,M]. */
double oracle_forward(const double* C, int N, int M, double gamma, double* R)
{
    const size_t W = (size_t)M + 1;
    for (size_t k = 0; k < ((size_t)N + 1) * W; ++k) R[k] = INFINITY;
    R[0] = 0.0;
    for (int i = 1; i <= N; ++i)
        for (int j = 1; j <= M; ++j) {
            double p[3] = { R[(i - 1) * W + (j - 1)], R[(i - 1) * W + j], R[i * W + (j - 1)] };
            double m = INFINITY;
            for (int q = 0; q < 3; ++q) if (p[q] < m) m = p[q];
            double s = 0.0;
            for (int q = 0; q < 3; ++q)
                if (isfinite(p[q])) s += exp(-(p[q] - m) / gamma);
            R[i * W + j] = C[(size_t)(i - 1) * M + (j - 1)] + m - gamma * log(s);
        }
    return R[(size_t)N * W + M];
}

/* E (N,M) from C and the R of oracle_forward. */
void oracle_backward(const double* C, const double* R, int N, int M, double gamma, double* E)
{
    const size_t W = (size_t)M + 1;
    /* E holds logE while the recursion runs, then is exponentiated. */
    for (int i = N; i >= 1; --i)
        for (int j = M; j >= 1; --j) {
            if (i == N && j == M) { E[(size_t)(N - 1) * M + (M - 1)] = 0.0; continue; }
            const double r = R[i * W + j];
            double t[3];
            int n = 0;
            const int si[3] = { i + 1, i, i + 1 };
            const int sj[3] = { j, j + 1, j + 1 };
            for (int q = 0; q < 3; ++q) {
                if (si[q] > N || sj[q] > M) continue;
                const size_t s = (size_t)(si[q] - 1) * M + (sj[q] - 1);
                t[n++] = E[s] + (R[si[q] * W + sj[q]] - C[s] - r) / gamma;
            }
            double mx = t[0];
            for (int q = 1; q < n; ++q) if (t[q] > mx) mx = t[q];
            double acc = 0.0;
            for (int q = 0; q < n; ++q) acc += exp(t[q] - mx);
            E[(size_t)(i - 1) * M + (j - 1)] = mx + log(acc);
        }
    for (size_t k = 0; k < (size_t)N * M; ++k) E[k] = exp(E[k]);
}

/* grad_x (N,D), grad_y (M,D); either may be NULL. */
void oracle_grads(const double* x, const double* y, const double* E, int N, int M, int D,
                  double g, double* gx, double* gy)
{
    if (gx) for (int i = 0; i < N; ++i)
        for (int k = 0; k < D; ++k) {
            double acc = 0.0;
            for (int j = 0; j < M; ++j)
                acc += E[(size_t)i * M + j] * (x[(size_t)i * D + k] - y[(size_t)j * D + k]);
            gx[(size_t)i * D + k] = 2.0 * g * acc;
        }
    if (gy) for (int j = 0; j < M; ++j)
        for (int k = 0; k < D; ++k) {
            double acc = 0.0;
            for (int i = 0; i < N; ++i)
                acc += E[(size_t)i * M + j] * (y[(size_t)j * D + k] - x[(size_t)i * D + k]);
            gy[(size_t)j * D + k] = 2.0 * g * acc;
        }
}

/* One problem end to end. R_out ((N+1)(M+1)) and E_out (N,M) may be NULL. */
int oracle_single(const double* x, const double* y, int N, int M, int D, double gamma,
                  double g, double* loss, double* gx, double* gy, double* R_out, double* E_out)
{
    if (N < 1 || M < 1 || D < 1 || !(gamma > 0.0)) return -1;
    double* C = (double*)malloc(sizeof(double) * (size_t)N * M);
    double* R = R_out ? R_out : (double*)malloc(sizeof(double) * ((size_t)N + 1) * ((size_t)M + 1));
    double* E = E_out ? E_out : (double*)malloc(sizeof(double) * (size_t)N * M);
    if (!C || !R || !E) {
        free(C);
        if (!R_out) free(R);
        if (!E_out) free(E);
        return -1;
    }
    oracle_sqeuclid(x, y, N, M, D, C);
    double v = oracle_forward(C, N, M, gamma, R);
    if (loss) *loss = v;
    if (gx || gy || E_out) {
        oracle_backward(C, R, N, M, gamma, E);
        oracle_grads(x, y, E, N, M, D, g, gx, gy);
    }
    free(C);
    if (!R_out) free(R);
    if (!E_out) free(E);
    return 0;
}

/* ---- batched ------------------------------------------------------------- */

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_threads_used(int nthreads)
{
#ifdef _OPENMP
    set_threads(nthreads);
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    (void)nthreads;
    return 1;
#endif
}

/* B independent problems. grad_loss NULL -> no gradients; gx/gy may be NULL. */
int oracle_batch(const double* x, const double* y, int B, int N, int M, int D, double gamma,
                 const double* grad_loss, double* loss, double* gx, double* gy, int nthreads)
{
    if (B < 1) return -1;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        const double g = grad_loss ? grad_loss[b] : 0.0;
        int rc = oracle_single(x + (size_t)b * N * D, y + (size_t)b * M * D, N, M, D, gamma, g,
                               loss ? loss + b : NULL,
                               (grad_loss && gx) ? gx + (size_t)b * N * D : NULL,
                               (grad_loss && gy) ? gy + (size_t)b * M * D : NULL, NULL, NULL);
        bad |= (rc != 0);
    }
    return bad ? -1 : 0;
}

/* Normalized Soft-DTW over B pairs of equal shape (N,D). */
int oracle_normalized(const double* x, const double* y, int B, int N, int D, double gamma,
                      const double* grad_loss, double* loss, double* gx, double* gy, int nthreads)
{
    if (B < 1 || N < 1 || D < 1) return -1;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        const double* xb = x + (size_t)b * N * D;
        const double* yb = y + (size_t)b * N * D;
        const double g = grad_loss ? grad_loss[b] : 0.0;
        const size_t n = (size_t)N * D;
        double* buf = (double*)malloc(sizeof(double) * 6 * n);
        if (!buf) { bad = 1; continue; }
        double *gxy_x = buf, *gxy_y = buf + n, *gxx_a = buf + 2 * n, *gxx_b = buf + 3 * n,
               *gyy_a = buf + 4 * n, *gyy_b = buf + 5 * n;
        double sxy, sxx, syy;
        int rc = oracle_single(xb, yb, N, N, D, gamma, 1.0, &sxy, gxy_x, gxy_y, NULL, NULL);
        rc |= oracle_single(xb, xb, N, N, D, gamma, 1.0, &sxx, gxx_a, gxx_b, NULL, NULL);
        rc |= oracle_single(yb, yb, N, N, D, gamma, 1.0, &syy, gyy_a, gyy_b, NULL, NULL);
        if (rc) { bad = 1; free(buf); continue; }
        if (loss) loss[b] = sxy - 0.5 * (sxx + syy);
        if (grad_loss) {
            for (size_t q = 0; q < n; ++q) {
                if (gx) gx[(size_t)b * n + q] = g * (gxy_x[q] - 0.5 * (gxx_a[q] + gxx_b[q]));
                if (gy) gy[(size_t)b * n + q] = g * (gxy_y[q] - 0.5 * (gyy_a[q] + gyy_b[q]));
            }
        }
        free(buf);
    }
    return bad ? -1 : 0;
}

/* One Adam step of the barycenter z (T,D) against X (K,T2,D). z, m, v updated
 * in place; t is the 1-based step number. loss_out (nullable) receives the
 * objective at the incoming z. grad_out (nullable, (T,D)) receives its gradient. */
/* One Adam step of the barycenter. max_grad_norm > 0 clips the gradient by its
 * global L2 norm first (SoftDTW README, "Time Series Barycenters": gradient
 * clipping; scale min(1, max_grad_norm / ||g||)); grad_out receives the raw,
 * unclipped gradient. */
int oracle_barycenter_step(double* z, double* m, double* v, int t, const double* X, int K,
                           int T, int T2, int D, double gamma, double lr, double b1, double b2,
                           double eps, double max_grad_norm, double* loss_out, double* grad_out, int nthreads)
{
    if (K < 1 || T < 1 || T2 < 1 || D < 1 || t < 1) return -1;
    const size_t n = (size_t)T * D;
    double* zs = (double*)malloc(sizeof(double) * n * K);
    double* gz = (double*)malloc(sizeof(double) * n * K);
    double* ls = (double*)malloc(sizeof(double) * K);
    double* gl = (double*)malloc(sizeof(double) * K);
    if (!zs || !gz || !ls || !gl) { free(zs); free(gz); free(ls); free(gl); return -1; }
    for (int k = 0; k < K; ++k) {
        memcpy(zs + (size_t)k * n, z, sizeof(double) * n);
        gl[k] = 1.0 / K;
    }
    int rc = oracle_batch(zs, X, K, T, T2, D, gamma, gl, ls, gz, NULL, nthreads);
    if (rc == 0) {
        double L = 0.0;
        for (int k = 0; k < K; ++k) L += ls[k];
        if (loss_out) *loss_out = L / K;
        const double c1 = 1.0 - pow(b1, t), c2 = 1.0 - pow(b2, t);
        double nrm2 = 0.0;
        for (size_t q = 0; q < n; ++q) {
            double g = 0.0;
            for (int k = 0; k < K; ++k) g += gz[(size_t)k * n + q];
            gz[q] = g;  /* part 0 now holds the summed gradient */
            nrm2 += g * g;
        }
        const double nrm = sqrt(nrm2);
        const double scale = (max_grad_norm > 0.0 && nrm > max_grad_norm) ? max_grad_norm / nrm : 1.0;
        for (size_t q = 0; q < n; ++q) {
            const double g = gz[q] * scale;
            if (grad_out) grad_out[q] = gz[q];
            m[q] = b1 * m[q] + (1.0 - b1) * g;
            v[q] = b2 * v[q] + (1.0 - b2) * g * g;
            z[q] -= lr * (m[q] / c1) / (sqrt(v[q] / c2) + eps);
        }
    }
    free(zs); free(gz); free(ls); free(gl);
    return rc;
}
