/*
 * lora_oracle.c -- plain fp64 CPU oracle of the LoRA linear layer.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline may load this file's library.  It shares no code, header, table or
 * helper with the CUDA path and must never be used as a fallback for it.
 *
 * What it computes, written as the plain definition:
 *
 *   Forward (ch05 "Acceleration principles: Triton kernels and fused LoRA",
 *   §5.3, LoRA equation y = W x + (alpha/r) B A x; the same map as
 *   ch01 "Project background", §1.2, y = W x + dW x with dW = (alpha/r) B A),
 *   applied to every token row of X (row-major, one token per row):
 *
 *       s = alpha / r
 *       H[m][i] = sum_k X[m][k] * A[i][k]                       H = X A^T
 *       Y[m][o] = sum_k X[m][k] * W[o][k] + s * sum_i H[m][i] * B[o][i]
 *
 *   Backward (ch05, §5.3 "the backward is fused too": gradients w.r.t.
 *   X, W (only if trained), A and B).  W is frozen, so no dW.  With the loss
 *   L = <dY, Y> (dY is the upstream gradient), differentiating the forward:
 *
 *       G[m][i]  = sum_o dY[m][o] * B[o][i]                     G = dY B
 *       dX[m][k] = sum_o dY[m][o] * W[o][k] + s * sum_i G[m][i] * A[i][k]
 *       dA[i][k] = s * sum_m G[m][i] * X[m][k]
 *       dB[o][i] = s * sum_m dY[m][o] * H[m][i]
 *
 * Every sum runs in increasing index order in double precision with no
 * blocking, so each output element has exactly one value whether it is
 * computed by the full routines or by the sampled ones.  Build with
 * -ffp-contract=off so that the result does not depend on FMA contraction.
 *
 * Layouts: X [M][d_in], W [d_out][d_in], A [r][d_in], B [d_out][r],
 * dY [M][d_out], H and G [M][r], all row-major, contiguous, double.
 */
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- one element of each quantity -------------------------------------- */

static double h_elem(const double *X, const double *A, int64_t d_in,
                     int64_t m, int64_t i)
{
    double acc = 0.0;
    for (int64_t k = 0; k < d_in; ++k)
        acc += X[m * d_in + k] * A[i * d_in + k];
    return acc;
}

static double g_elem(const double *dY, const double *B, int64_t d_out,
                     int64_t r, int64_t m, int64_t i)
{
    double acc = 0.0;
    for (int64_t o = 0; o < d_out; ++o)
        acc += dY[m * d_out + o] * B[o * r + i];
    return acc;
}

static double y_elem(const double *X, const double *W, const double *B,
                     const double *H, double s, int64_t d_in, int64_t r,
                     int64_t m, int64_t o)
{
    double base = 0.0;
    for (int64_t k = 0; k < d_in; ++k)
        base += X[m * d_in + k] * W[o * d_in + k];
    double low = 0.0;
    for (int64_t i = 0; i < r; ++i)
        low += H[m * r + i] * B[o * r + i];
    return base + s * low;
}

static double dx_elem(const double *dY, const double *W, const double *A,
                      const double *G, double s, int64_t d_in, int64_t d_out,
                      int64_t r, int64_t m, int64_t k)
{
    double base = 0.0;
    for (int64_t o = 0; o < d_out; ++o)
        base += dY[m * d_out + o] * W[o * d_in + k];
    double low = 0.0;
    for (int64_t i = 0; i < r; ++i)
        low += G[m * r + i] * A[i * d_in + k];
    return base + s * low;
}

static double da_elem(const double *G, const double *X, double s, int64_t M,
                      int64_t d_in, int64_t r, int64_t i, int64_t k)
{
    double acc = 0.0;
    for (int64_t m = 0; m < M; ++m)
        acc += G[m * r + i] * X[m * d_in + k];
    return s * acc;
}

static double db_elem(const double *dY, const double *H, double s, int64_t M,
                      int64_t d_out, int64_t r, int64_t o, int64_t i)
{
    double acc = 0.0;
    for (int64_t m = 0; m < M; ++m)
        acc += dY[m * d_out + o] * H[m * r + i];
    return s * acc;
}

/* ---- full tensors -------------------------------------------------------- */

int lora_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* H = X A^T, [M][r] */
void lora_oracle_h(const double *X, const double *A, int64_t M, int64_t d_in,
                   int64_t r, double *H)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < r; ++i)
            H[m * r + i] = h_elem(X, A, d_in, m, i);
}

/* G = dY B, [M][r] */
void lora_oracle_g(const double *dY, const double *B, int64_t M, int64_t d_out,
                   int64_t r, double *G)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < r; ++i)
            G[m * r + i] = g_elem(dY, B, d_out, r, m, i);
}

/* Y = X W^T + s H B^T, [M][d_out]; H from lora_oracle_h */
void lora_oracle_y(const double *X, const double *W, const double *B,
                   const double *H, double s, int64_t M, int64_t d_in,
                   int64_t d_out, int64_t r, double *Y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t o = 0; o < d_out; ++o)
            Y[m * d_out + o] = y_elem(X, W, B, H, s, d_in, r, m, o);
}

/* dX = dY W + s G A, [M][d_in]; G from lora_oracle_g */
void lora_oracle_dx(const double *dY, const double *W, const double *A,
                    const double *G, double s, int64_t M, int64_t d_in,
                    int64_t d_out, int64_t r, double *dX)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < d_in; ++k)
            dX[m * d_in + k] = dx_elem(dY, W, A, G, s, d_in, d_out, r, m, k);
}

/* dA = s G^T X, [r][d_in] */
void lora_oracle_da(const double *G, const double *X, double s, int64_t M,
                    int64_t d_in, int64_t r, double *dA)
{
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < d_in; ++k)
        for (int64_t i = 0; i < r; ++i)
            dA[i * d_in + k] = da_elem(G, X, s, M, d_in, r, i, k);
}

/* dB = s dY^T H, [d_out][r] */
void lora_oracle_db(const double *dY, const double *H, double s, int64_t M,
                    int64_t d_out, int64_t r, double *dB)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < d_out; ++o)
        for (int64_t i = 0; i < r; ++i)
            dB[o * r + i] = db_elem(dY, H, s, M, d_out, r, o, i);
}

/* ---- sampled elements (same per-element sums as above) ------------------ */

/* H[:, i] for one column i: out[M] */
void lora_oracle_h_col(const double *X, const double *A, int64_t M,
                       int64_t d_in, int64_t i, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        out[m] = h_elem(X, A, d_in, m, i);
}

/* G[:, i] for one column i: out[M] */
void lora_oracle_g_col(const double *dY, const double *B, int64_t M,
                       int64_t d_out, int64_t r, int64_t i, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        out[m] = g_elem(dY, B, d_out, r, m, i);
}

/* Rows rows[j] of H and of G, written in place into full-size [M][r]
 * arrays (other rows are left untouched). */
void lora_oracle_h_rows(const double *X, const double *A, int64_t d_in,
                        int64_t r, const int64_t *rows, int64_t n_rows,
                        double *H)
{
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t j = 0; j < n_rows; ++j)
        for (int64_t i = 0; i < r; ++i)
            H[rows[j] * r + i] = h_elem(X, A, d_in, rows[j], i);
}

void lora_oracle_g_rows(const double *dY, const double *B, int64_t d_out,
                        int64_t r, const int64_t *rows, int64_t n_rows,
                        double *G)
{
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t j = 0; j < n_rows; ++j)
        for (int64_t i = 0; i < r; ++i)
            G[rows[j] * r + i] = g_elem(dY, B, d_out, r, rows[j], i);
}

/* Y[rows[j]][:] for n_rows rows, out [n_rows][d_out].  H holds the full
 * [M][r] matrix or one filled by lora_oracle_h_rows for the sampled rows. */
void lora_oracle_y_rows(const double *X, const double *W, const double *B,
                        const double *H, double s, int64_t d_in,
                        int64_t d_out, int64_t r, const int64_t *rows,
                        int64_t n_rows, double *out)
{
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t j = 0; j < n_rows; ++j)
        for (int64_t o = 0; o < d_out; ++o)
            out[j * d_out + o] = y_elem(X, W, B, H, s, d_in, r, rows[j], o);
}

/* dX[rows[j]][:] for n_rows rows, out [n_rows][d_in] */
void lora_oracle_dx_rows(const double *dY, const double *W, const double *A,
                         const double *G, double s, int64_t d_in,
                         int64_t d_out, int64_t r, const int64_t *rows,
                         int64_t n_rows, double *out)
{
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t j = 0; j < n_rows; ++j)
        for (int64_t k = 0; k < d_in; ++k)
            out[j * d_in + k] =
                dx_elem(dY, W, A, G, s, d_in, d_out, r, rows[j], k);
}

/* dA[i][k] for the pairs (ii[j], kk[j]).  gcols holds, for each pair, the
 * full column G[:, ii[j]] as gcols[j*M .. j*M+M) (from lora_oracle_g_col);
 * it is read through a one-column view so that the sum is da_elem's. */
void lora_oracle_da_entries(const double *gcols, const double *X, double s,
                            int64_t M, int64_t d_in, const int64_t *kk,
                            int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = da_elem(gcols + j * M, X, s, M, d_in, 1, 0, kk[j]);
}

/* dB[o][i] for the pairs (oo[j], ii[j]); hcols[j*M ..] = H[:, ii[j]] */
void lora_oracle_db_entries(const double *dY, const double *hcols, double s,
                            int64_t M, int64_t d_out, const int64_t *oo,
                            int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = db_elem(dY, hcols + j * M, s, M, d_out, 1, oo[j], 0);
}
