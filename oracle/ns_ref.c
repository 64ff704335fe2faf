/*
 * Plain C, double-precision, triple-loop Newton–Schulz (TEST INFRASTRUCTURE).
 *
 * A third, BLAS-free statement of the iteration of "Muon 优化器"
 * (DeepSeek-V4 tech notes) §2 "Hybrid Newton–Schulz 正交化":
 *   X0 = X / ||X||_F  (zero input returned unchanged),
 *   X_{k} = a X + b (X X^T) X + c (X X^T)^2 X.
 * It always forms the Gram on the row side, whatever the shape, so for tall
 * inputs it also checks the transpose reading of the NumPy oracle.  Meant for
 * tiny matrices (O(rows^2 * cols) per step).  Only the tests call it; the
 * CUDA library neither links nor includes it.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* out[r x c] = a * x[r x k] @ y[k x c]  (row-major) */
static void matmul(const double* x, const double* y, double* out, int r, int k, int c) {
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) {
            double s = 0.0;
            for (int t = 0; t < k; ++t) s += x[(size_t)i * k + t] * y[(size_t)t * c + j];
            out[(size_t)i * c + j] = s;
        }
}

/* coeffs: iters x 3 (a, b, c).  Returns 0 on success, -1 on bad arguments or
 * allocation failure. */
int ns_ref_iterate(const double* x, int rows, int cols, const double* coeffs, int iters,
                   int normalize, double* out) {
    if (!x || !out || rows < 1 || cols < 1 || iters < 0 || (iters > 0 && !coeffs)) return -1;
    size_t n = (size_t)rows * cols;
    double* S = (double*)malloc(sizeof(double) * (size_t)rows * rows);
    double* SX = (double*)malloc(sizeof(double) * n);
    double* SSX = (double*)malloc(sizeof(double) * n);
    double* Xt = (double*)malloc(sizeof(double) * n);
    if (!S || !SX || !SSX || !Xt) { free(S); free(SX); free(SSX); free(Xt); return -1; }
    memcpy(out, x, sizeof(double) * n);
    if (normalize) {
        double ss = 0.0;
        for (size_t i = 0; i < n; ++i) ss += out[i] * out[i];
        if (ss == 0.0) { free(S); free(SX); free(SSX); free(Xt); return 0; }
        double inv = 1.0 / sqrt(ss);
        for (size_t i = 0; i < n; ++i) out[i] *= inv;
    }
    for (int it = 0; it < iters; ++it) {
        double a = coeffs[3 * it + 0], b = coeffs[3 * it + 1], c = coeffs[3 * it + 2];
        /* Xt = X^T (cols x rows), S = X X^T (rows x rows) */
        for (int i = 0; i < rows; ++i)
            for (int j = 0; j < cols; ++j) Xt[(size_t)j * rows + i] = out[(size_t)i * cols + j];
        matmul(out, Xt, S, rows, cols, rows);
        matmul(S, out, SX, rows, rows, cols);
        matmul(S, SX, SSX, rows, rows, cols);
        for (size_t i = 0; i < n; ++i) out[i] = a * out[i] + b * SX[i] + c * SSX[i];
    }
    free(S); free(SX); free(SSX); free(Xt);
    return 0;
}
