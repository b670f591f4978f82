/*
 * Oracle: plain, slow, obviously correct forward 2-D convolution in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of the convolution the surveyed
 * pages turn on ("GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a
 * Custom PyTorch Extension", sections "Where the Performance Bottleneck
 * Appeared" -- nested loops over input channels, output filters, spatial
 * positions, kernel dimensions and batch -- and "Transforming Conv2D into
 * im2col and GEMM", where each output is a weight row times an unflipped input
 * window; "Enabling Memory-efficient Im2win Convolution ...", abstract):
 *
 *   y[n,k,p,q] = bias[k] + sum_{c,r,s} x[n, c, p*stride - pad + r*dil,
 *                                            q*stride - pad + s*dil] * w[k,c,r,s]
 *
 * with x read as zero outside 0 <= h < H, 0 <= w < W (zero padding), no
 * kernel flip (cross-correlation), and
 *
 *   P = floor((H + 2*pad - dil*(R-1) - 1) / stride) + 1   (Q likewise from W, S).
 *
 * Besides y it returns den[n,k,p,q] = |bias[k]| + sum |x|*|w| over the same
 * in-range taps; the parity tests divide |y_gpu - y| by it.
 *
 * Layouts here are fixed: x is [N][C][H][W], w is [K][C][R][S], y and den are
 * [N][K][P][Q], all fp64 and contiguous.  Callers convert other layouts and
 * dtypes to this form exactly before calling (a permutation and an exact
 * widening, no arithmetic).  bias may be NULL (read as zero).
 *
 * Work is split over (n, k) with OpenMP; each output is accumulated by one
 * thread in the fixed order c, r, s, so the result does not depend on the
 * thread count.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Output extent along one axis; <= 0 means the shape is invalid. */
int64_t oracle_out_extent(int64_t in, int64_t ksize, int64_t stride, int64_t pad, int64_t dil)
{
    if (in < 1 || ksize < 1 || stride < 1 || pad < 0 || dil < 1) return 0;
    int64_t span = in + 2 * pad - dil * (ksize - 1) - 1;
    if (span < 0) return 0;
    return span / stride + 1;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One output element of the definition above. */
static void one_output(const double *x, const double *w, const double *bias,
                       int64_t C, int64_t H, int64_t W, int64_t R, int64_t S,
                       int64_t stride, int64_t pad, int64_t dil,
                       int64_t n, int64_t k, int64_t p, int64_t q,
                       double *y_out, double *den_out)
{
    double acc = bias ? bias[k] : 0.0;
    double den = bias ? fabs(bias[k]) : 0.0;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t r = 0; r < R; ++r) {
            int64_t h = p * stride - pad + r * dil;
            if (h < 0 || h >= H) continue;
            for (int64_t s = 0; s < S; ++s) {
                int64_t ww = q * stride - pad + s * dil;
                if (ww < 0 || ww >= W) continue;
                double xv = x[((n * C + c) * H + h) * W + ww];
                double wv = w[((k * C + c) * R + r) * S + s];
                acc += xv * wv;
                den += fabs(xv) * fabs(wv);
            }
        }
    }
    *y_out = acc;
    if (den_out) *den_out = den;
}

/*
 * Full output.  threads <= 0 uses the OpenMP default.  Returns 0, or -1 when a
 * size is invalid (the output is then untouched).
 */
int oracle_conv2d_f64(const double *x, const double *w, const double *bias,
                      double *y, double *den,
                      int64_t N, int64_t C, int64_t H, int64_t W,
                      int64_t K, int64_t R, int64_t S,
                      int64_t stride, int64_t pad, int64_t dil, int threads)
{
    if (N < 1 || C < 1 || K < 1) return -1;
    int64_t P = oracle_out_extent(H, R, stride, pad, dil);
    int64_t Q = oracle_out_extent(W, S, stride, pad, dil);
    if (P < 1 || Q < 1) return -1;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
    int64_t NK = N * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t nk = 0; nk < NK; ++nk) {
        int64_t n = nk / K, k = nk % K;
        for (int64_t p = 0; p < P; ++p)
            for (int64_t q = 0; q < Q; ++q) {
                int64_t o = ((n * K + k) * P + p) * Q + q;
                one_output(x, w, bias, C, H, W, R, S, stride, pad, dil, n, k, p, q,
                           &y[o], den ? &den[o] : NULL);
            }
    }
    return 0;
}

/*
 * Selected outputs only: idx holds count quadruples (n, k, p, q); y[i] and
 * den[i] receive output i.  Returns 0, -1 for an invalid size, -2 for an index
 * out of range.
 */
int oracle_conv2d_f64_points(const double *x, const double *w, const double *bias,
                             const int64_t *idx, int64_t count, double *y, double *den,
                             int64_t N, int64_t C, int64_t H, int64_t W,
                             int64_t K, int64_t R, int64_t S,
                             int64_t stride, int64_t pad, int64_t dil, int threads)
{
    if (N < 1 || C < 1 || K < 1) return -1;
    int64_t P = oracle_out_extent(H, R, stride, pad, dil);
    int64_t Q = oracle_out_extent(W, S, stride, pad, dil);
    if (P < 1 || Q < 1) return -1;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t *t = idx + 4 * i;
        if (t[0] < 0 || t[0] >= N || t[1] < 0 || t[1] >= K ||
            t[2] < 0 || t[2] >= P || t[3] < 0 || t[3] >= Q) return -2;
    }
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t *t = idx + 4 * i;
        one_output(x, w, bias, C, H, W, R, S, stride, pad, dil, t[0], t[1], t[2], t[3],
                   &y[i], den ? &den[i] : NULL);
    }
    return 0;
}
