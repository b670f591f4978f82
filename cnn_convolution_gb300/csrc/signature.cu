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
// One CTA per end time.  A thread owns one window and a 2x2 block of
// (i, j) pairs -- rows i0, i0+1 against columns j0, j0+1, blocks with
// j0 >= i0 only: the matrices are symmetric (s_i s_j = s_j s_i exactly), so
// an off-diagonal block is also written transposed.  The end time's samples
// (its longest window) are staged once in shared memory by asynchronous
// copies, time-major ([position][signal], so one 8-byte read gives a signal
// pair at one time step); windows too long for shared memory are read
// through the read-only cache instead.  Each thread runs one plain loop over
// its window, newest sample first: two 8-byte reads feed 4 FMAs into 4
// fp32 accumulators that start from zero, then divides each by w once.
// Threads of a warp share one window (the block count is padded to a
// multiple of 32), so a warp's loop has one trip count.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kSigThreads = 384;
constexpr int kSigMaxWindows = 8;
constexpr int kSigSmemMax = 96 * 1024;   // larger windows are read from global memory

struct SigParams {
    const float *series;   // [n][T]
    float *out;            // [n_steps][n_windows][n][n]
    int n, T, n_win, t_first, wmax;
    int sstride;           // staged floats per position: >= n rounded up to even, = 2 mod 32
    int nblk, nblk_pad;    // 2x2 blocks with j0 >= i0; that count rounded up to a multiple of 32
    int win[kSigMaxWindows];
};

// Signals i, i + 1 at one position; a signal index >= n reads as 0.
template <bool kStaged>
__device__ __forceinline__ float2 sig_pair(const float *ss, const SigParams &p, int64_t t_lo, int i, int pos) {
    if constexpr (kStaged) {
        return *reinterpret_cast<const float2 *>(ss + pos * p.sstride + i);
    } else {
        const float *g = p.series + t_lo + pos + (int64_t)i * p.T;
        return make_float2(__ldg(g), i + 1 < p.n ? __ldg(g + p.T) : 0.f);
    }
}

// Positions index the end time's samples: position 0 is time e - wmax, the
// newest sample e - 1 is position wmax - 1; window w reads wmax - w .. wmax - 1.
template <bool kStaged>
__global__ void __launch_bounds__(kSigThreads) signature_kernel(const __grid_constant__ SigParams p) {
    extern __shared__ __align__(16) float ss[];   // [position][sstride]
    // no early trigger: a kernel of many short CTAs lets the next one launch
    // at its exit, so the next grid is spread over idle SMs
    sm103a::pdl_wait();                        // the previous kernel's writes are visible
    const int b = blockIdx.x;
    const int64_t t_lo = (int64_t)p.t_first + b - p.wmax;
    const int n_pad = (p.n + 1) & ~1;
    if constexpr (kStaged) {
        // one signal per warp at a time, consecutive positions across the
        // lanes (coalesced reads); every copy in flight before the wait
        const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
        const uint32_t ss_u = sm103a::smem_u32(ss);
        for (int i = warp; i < n_pad; i += kSigThreads / 32) {
            const float *row = p.series + (int64_t)min(i, p.n - 1) * p.T + t_lo;
            for (int q = lane; q < p.wmax; q += 32)
                sm103a::cp_async_f32(ss_u + 4u * (uint32_t)(q * p.sstride + i), row + q, i < p.n);
        }
        sm103a::cp_async_commit();
        sm103a::cp_async_wait<0>();
    }
    __syncthreads();

    const int item = blockIdx.y * kSigThreads + (int)threadIdx.x;
    const int c = item / p.nblk_pad, k = item - c * p.nblk_pad;
    if (c >= p.n_win || k >= p.nblk) return;
    // block k -> (bi, bj), bi <= bj, rows of the upper triangle in order:
    // row bi starts at S(bi) = bi*nt - bi(bi-1)/2; the root of S(x) = k,
    // then at most one step to correct its rounding
    const int nt = n_pad / 2;
    const int e2 = 2 * nt + 1;
    int bi = (int)(((float)e2 - sqrtf((float)(e2 * e2 - 8 * k))) * 0.5f);
    bi = max(0, min(bi, nt - 1));
    if (bi > 0 && k < bi * nt - bi * (bi - 1) / 2) --bi;
    if (bi + 1 < nt && k >= (bi + 1) * nt - (bi + 1) * bi / 2) ++bi;
    const int i0 = 2 * bi, j0 = 2 * (bi + k - (bi * nt - bi * (bi - 1) / 2));

    const int w = p.win[c];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};     // pair (i0 + u / 2, j0 + u % 2)
#pragma unroll 4
    for (int pos = p.wmax - 1; pos >= p.wmax - w; --pos) {
        const float2 a = sig_pair<kStaged>(ss, p, t_lo, i0, pos);
        const float2 v = sig_pair<kStaged>(ss, p, t_lo, j0, pos);
        acc[0] = fmaf(a.x, v.x, acc[0]);
        acc[1] = fmaf(a.x, v.y, acc[1]);
        acc[2] = fmaf(a.y, v.x, acc[2]);
        acc[3] = fmaf(a.y, v.y, acc[3]);
    }
    float *o = p.out + ((int64_t)b * p.n_win + c) * p.n * p.n;
    const float wf = (float)w;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = i0 + u / 2, j = j0 + u % 2;
        if (i < p.n && j < p.n) {
            const float m = acc[u] / wf;
            o[i * p.n + j] = m;
            if (i0 != j0) o[j * p.n + i] = m;   // a diagonal block holds both (i, j) and (j, i)
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
    p.wmax = 0;
    for (int c = 0; c < n_windows; ++c) {
        p.win[c] = windows[c];
        p.wmax = std::max(p.wmax, windows[c]);
    }
    const int n_pad = (n + 1) & ~1;
    // = 2 mod 32: the staging writes (lanes on consecutive positions) spread over 16 banks
    p.sstride = n_pad + (34 - n_pad % 32) % 32;
    const int nt = n_pad / 2;
    p.nblk = nt * (nt + 1) / 2;
    p.nblk_pad = (p.nblk + 31) / 32 * 32;
    const size_t smem = (size_t)p.wmax * p.sstride * sizeof(float);
    const bool staged = smem <= (size_t)kSigSmemMax;
    const int items = n_windows * p.nblk_pad;
    const dim3 grid((unsigned)n_steps, (unsigned)((items + kSigThreads - 1) / kSigThreads));
    cudaError_t e;
    if (staged) {
        if (smem > 48 * 1024) {
            // the attribute once per device: setting it on every call stalls the host
            static std::atomic<uint64_t> attr_done{0};
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
            const uint64_t bit = (uint64_t)1 << (dev & 63);
            if (!(attr_done.load(std::memory_order_acquire) & bit)) {
                if (cudaFuncSetAttribute(signature_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSigSmemMax) != cudaSuccess)
                    return CONV2D_ERR_CUDA;
                attr_done.fetch_or(bit, std::memory_order_release);
            }
        }
        e = launch_pdl(signature_kernel<true>, grid, dim3(kSigThreads), smem, st, p);
    } else {
        e = launch_pdl(signature_kernel<false>, grid, dim3(kSigThreads), 0, st, p);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

}  // namespace conv2d
