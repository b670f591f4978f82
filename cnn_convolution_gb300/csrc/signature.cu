// MSCRED signature matrices on the GPU, written straight into the NCHW input
// of the encoder's first convolution.
//
// "GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
// Extension" (section "Why Signature Matrices Are Useful"): a signature
// matrix holds the pairwise relationships of the signals over one time
// interval, at several interval lengths.  For signals s_i(t), end time e and
// window w (the definition of the MSCRED paper that page cites):
//
//     M_ij(e, w) = sum_{t = e-w}^{e-1} s_i(t) * s_j(t) / w
//
// out[b][c][i][j] = M_ij(t_first + b, windows[c]).
//
// One CTA per end time (grid.y splits the n*n pairs when there are more than
// one CTA's worth).  The samples are staged in shared memory in chunks of
// 64 time steps (rows padded to an odd stride, so the lanes of a warp, which
// read different signals at one time step, hit different banks), walked
// from the most recent backwards; because every window
// ends at e, the windows are nested, so one pass over the longest window
// emits every window's matrix as soon as its sample count is reached (the
// windows are visited in increasing length).  Each thread accumulates its
// pairs in fp32 with FMA in that fixed order and divides by w once.

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kSigThreads = 256;
constexpr int kSigChunk = 64;      // time steps staged per pass
constexpr int kSigStride = kSigChunk + 1;   // odd row stride: lanes reading different rows hit different banks
constexpr int kSigPairs = 4;       // (i, j) pairs per thread
constexpr int kSigMaxWindows = 8;

struct SigParams {
    const float *series;   // [n][T]
    float *out;            // [n_steps][n_windows][n][n]
    int n, T, n_win, t_first;
    int win[kSigMaxWindows];    // window lengths, increasing
    int chan[kSigMaxWindows];   // output channel of each
};

__global__ void __launch_bounds__(kSigThreads) signature_kernel(const SigParams p) {
    extern __shared__ float ss[];              // [n][kSigStride]
    // no early trigger: a kernel of many short CTAs lets the next one launch
    // at its exit, so the next grid is spread over idle SMs
    sm103a::pdl_wait();                        // the previous kernel's writes are visible
    const int b = blockIdx.x;
    const int e = p.t_first + b;
    const int nn = p.n * p.n;
    const int pid0 = blockIdx.y * (kSigThreads * kSigPairs) + (int)threadIdx.x;
    int pi[kSigPairs], pj[kSigPairs];
#pragma unroll
    for (int q = 0; q < kSigPairs; ++q) {
        const int pid = pid0 + q * kSigThreads;
        pi[q] = pid < nn ? pid / p.n : 0;
        pj[q] = pid < nn ? pid - pi[q] * p.n : 0;
    }
    float acc[kSigPairs];
#pragma unroll
    for (int q = 0; q < kSigPairs; ++q) acc[q] = 0.f;

    // the window table in shared memory; the next boundary stays in a register
    __shared__ int s_win[kSigMaxWindows], s_chan[kSigMaxWindows];
    if (threadIdx.x < kSigMaxWindows) {
        s_win[threadIdx.x] = threadIdx.x < (unsigned)p.n_win ? p.win[threadIdx.x] : 0;
        s_chan[threadIdx.x] = threadIdx.x < (unsigned)p.n_win ? p.chan[threadIdx.x] : 0;
    }
    __syncthreads();
    const int wmax = s_win[p.n_win - 1];
    int count = 0, next = 0;                   // samples summed so far, next window to emit
    int next_w = s_win[0];
    for (int t_hi = e; t_hi > e - wmax; t_hi -= kSigChunk) {
        const int len = min(kSigChunk, t_hi - (e - wmax));
        const int t_lo = t_hi - len;
        __syncthreads();                       // the previous chunk is no longer read
        // every load of the chunk is issued before any of them is stored
        for (int k0 = 0; k0 < p.n * len; k0 += kSigThreads * 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int k = k0 + u * kSigThreads + (int)threadIdx.x;
                const int i = k / len, tt = k - i * len;
                const bool in = k < p.n * len;
                v[u] = sm103a::ldg_or_zero(p.series + (in ? (int64_t)i * p.T + t_lo + tt : 0), in);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int k = k0 + u * kSigThreads + (int)threadIdx.x;
                const int i = k / len, tt = k - i * len;
                if (k < p.n * len) ss[i * kSigStride + tt] = v[u];
            }
        }
        __syncthreads();
        for (int tt = len - 1; tt >= 0; --tt) {
#pragma unroll
            for (int q = 0; q < kSigPairs; ++q)
                acc[q] = fmaf(ss[pi[q] * kSigStride + tt], ss[pj[q] * kSigStride + tt], acc[q]);
            ++count;
            while (count == next_w) {
                const float w = (float)next_w;
                float *o = p.out + ((int64_t)b * p.n_win + s_chan[next]) * nn;
#pragma unroll
                for (int q = 0; q < kSigPairs; ++q) {
                    const int pid = pid0 + q * kSigThreads;
                    if (pid < nn) o[pid] = acc[q] / w;
                }
                ++next;
                next_w = next < p.n_win ? s_win[next] : 0;
            }
        }
    }
}

}  // namespace

conv2d_status_t sig_launch(const float *series, int n, int T, const int *windows, int n_windows,
                           int t_first, int n_steps, float *out, cudaStream_t st) {
    SigParams p;
    p.series = series;
    p.out = out;
    p.n = n;
    p.T = T;
    p.n_win = n_windows;
    p.t_first = t_first;
    int order[kSigMaxWindows];
    for (int c = 0; c < n_windows; ++c) order[c] = c;
    std::sort(order, order + n_windows, [&](int a, int b) {
        return windows[a] < windows[b] || (windows[a] == windows[b] && a < b);
    });
    for (int c = 0; c < n_windows; ++c) {
        p.win[c] = windows[order[c]];
        p.chan[c] = order[c];
    }
    const int per_cta = kSigThreads * kSigPairs;
    const dim3 grid((unsigned)n_steps, (unsigned)((n * n + per_cta - 1) / per_cta));
    const size_t smem = (size_t)n * kSigStride * sizeof(float);
    if (launch_pdl(signature_kernel, grid, dim3(kSigThreads), smem, st, p) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

}  // namespace conv2d
