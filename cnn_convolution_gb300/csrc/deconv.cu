// Transposed convolution ("deconvolution") forward, fp32 NCHW: the MSCRED
// decoder's up-sampling layer.
//
// "GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
// Extension" (section "Understanding MSCRED": the decoder reconstructs the
// signature matrices).  The layer is the adjoint of the forward convolution
// in its input:
//
//   y[n,c,h,w] = bias[c] + sum over k and taps (r, s) with
//                h = p*stride - pad + r*dil, w = q*stride - pad + s*dil
//                of x[n,k,p,q] * wt[k,c,r,s]
//
// computed as a gather (no scatter, no atomics, deterministic): an output
// pixel takes tap r exactly when (h + pad - r*dil) is a multiple of the
// stride and p = (h + pad - r*dil) / stride lies in [0, P).
//
// A CTA of 256 threads owns an 8 x 32 block of output pixels of one image
// (warp = row, lane = column) and 32 output channels (registers).  For each
// chunk of 8 input channels it stages the input footprint of the block
// (zero outside x) and the chunk's weights as [k][r][s][32 channels] in
// shared memory.  A warp's row decides its valid filter rows uniformly; each
// lane keeps a bitmask of its valid filter columns.  Per valid tap: one
// input read, 8 broadcast 16-byte weight reads, 32 FFMAs.

#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kDvThreads = 256;
constexpr int kDvRows = 8, kDvCols = 32;
constexpr int kDvC = 32;             // output channels per CTA
constexpr int kDvK = 8;              // input channels per staged chunk
constexpr int kDvMaxTap = 8;         // R, S <= 8

struct DvParams {
    const float *x, *w, *bias;
    float *y;
    int N, K, P, Q, C, R, S, H, W;
    int stride, pad, dil;
    int tiles_h, tiles_w, c_blocks;
    int IP, IQ;                      // staged footprint rows / columns (upper bounds)
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

__global__ void __launch_bounds__(kDvThreads, 2) deconv_kernel(const DvParams p) {
    extern __shared__ float4 dv_smem4[];
    float *xs = reinterpret_cast<float *>(dv_smem4);                   // [kDvK][IP][IQ]
    const int xs_sz = (kDvK * p.IP * p.IQ + 3) & ~3;
    float *ws = xs + xs_sz;                                             // [kDvK][R][S][kDvC]

    int t = blockIdx.x;
    const int cb = t % p.c_blocks;
    t /= p.c_blocks;
    const int tw = t % p.tiles_w;
    t /= p.tiles_w;
    const int th = t % p.tiles_h;
    const int n = t / p.tiles_h;
    const int h0 = th * kDvRows, w0 = tw * kDvCols, c0 = cb * kDvC;
    // first input row / column the block can read
    const int p_lo = floor_div(h0 + p.pad - (p.R - 1) * p.dil + p.stride - 1, p.stride);
    const int q_lo = floor_div(w0 + p.pad - (p.S - 1) * p.dil + p.stride - 1, p.stride);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = h0 + warp, wcol = w0 + lane;
    // valid taps: rows (uniform in the warp), columns (per lane)
    unsigned rmask = 0, smask = 0;
    int pl[kDvMaxTap], ql[kDvMaxTap];
#pragma unroll
    for (int r = 0; r < kDvMaxTap; ++r) {
        pl[r] = 0;
        if (r < p.R) {
            const int hp = h + p.pad - r * p.dil;
            if (hp >= 0 && hp % p.stride == 0 && hp / p.stride < p.P) {
                rmask |= 1u << r;
                pl[r] = hp / p.stride - p_lo;
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kDvMaxTap; ++s) {
        ql[s] = 0;
        if (s < p.S) {
            const int wp = wcol + p.pad - s * p.dil;
            if (wp >= 0 && wp % p.stride == 0 && wp / p.stride < p.Q) {
                smask |= 1u << s;
                ql[s] = wp / p.stride - q_lo;
            }
        }
    }
    if (h >= p.H) rmask = 0;
    if (wcol >= p.W) smask = 0;

    float acc[kDvC];
#pragma unroll
    for (int j = 0; j < kDvC; ++j) acc[j] = 0.f;
    const int RS = p.R * p.S;
    const int xn = kDvK * p.IP * p.IQ, wn = kDvK * RS * kDvC;

    for (int k0 = 0; k0 < p.K; k0 += kDvK) {
        __syncthreads();
        for (int i = threadIdx.x; i < xn; i += kDvThreads) {
            const int iq = i % p.IQ;
            const int r2 = i / p.IQ;
            const int ip = r2 % p.IP;
            const int kk = r2 / p.IP;
            const int k = k0 + kk, pp = p_lo + ip, qq = q_lo + iq;
            const bool in = k < p.K && (unsigned)pp < (unsigned)p.P && (unsigned)qq < (unsigned)p.Q;
            const int64_t off = (((int64_t)n * p.K + k) * p.P + pp) * p.Q + qq;
            xs[i] = sm103a::ldg_or_zero(p.x + (in ? off : 0), in);
        }
        for (int i = threadIdx.x; i < wn; i += kDvThreads) {
            const int j = i % kDvC;
            const int r2 = i / kDvC;
            const int rs = r2 % RS;
            const int kk = r2 / RS;
            const int k = k0 + kk, c = c0 + j;
            const bool in = k < p.K && c < p.C;
            const int64_t off = ((int64_t)k * p.C + c) * RS + rs;
            ws[i] = sm103a::ldg_or_zero(p.w + (in ? off : 0), in);
        }
        __syncthreads();
        const int kn = min(kDvK, p.K - k0);
        for (int kk = 0; kk < kn; ++kk) {
            const float *xk = xs + kk * p.IP * p.IQ;
            const float *wk = ws + kk * RS * kDvC;
#pragma unroll
            for (int r = 0; r < kDvMaxTap; ++r) {
                if (!((rmask >> r) & 1u)) continue;
                const float *xr = xk + pl[r] * p.IQ;
#pragma unroll
                for (int s = 0; s < kDvMaxTap; ++s) {
                    if (!((smask >> s) & 1u)) continue;
                    const float a = xr[ql[s]];
                    const float4 *w4 = reinterpret_cast<const float4 *>(wk + (r * p.S + s) * kDvC);
#pragma unroll
                    for (int j = 0; j < kDvC / 4; ++j) {
                        const float4 v = w4[j];
                        acc[4 * j] = fmaf(a, v.x, acc[4 * j]);
                        acc[4 * j + 1] = fmaf(a, v.y, acc[4 * j + 1]);
                        acc[4 * j + 2] = fmaf(a, v.z, acc[4 * j + 2]);
                        acc[4 * j + 3] = fmaf(a, v.w, acc[4 * j + 3]);
                    }
                }
            }
        }
    }
    if (h >= p.H || wcol >= p.W) return;
    const int64_t HW = (int64_t)p.H * p.W;
    float *yp = p.y + ((int64_t)n * p.C + c0) * HW + (int64_t)h * p.W + wcol;
#pragma unroll
    for (int j = 0; j < kDvC; ++j) {
        if (c0 + j < p.C) yp[(int64_t)j * HW] = acc[j] + (p.bias ? __ldg(p.bias + c0 + j) : 0.f);
    }
}

void footprint(int stride, int dil, int R, int S, int *ip, int *iq) {
    // rows of x a block of kDvRows output rows can read (an upper bound)
    *ip = (kDvRows - 1 + (R - 1) * dil) / stride + 2;
    *iq = (kDvCols - 1 + (S - 1) * dil) / stride + 2;
}

}  // namespace

size_t dv_smem_bytes(int stride, int dil, int R, int S) {
    int ip, iq;
    footprint(stride, dil, R, S, &ip, &iq);
    const size_t xs = ((size_t)kDvK * ip * iq + 3) & ~(size_t)3;
    return (xs + (size_t)kDvK * R * S * kDvC) * sizeof(float);
}

conv2d_status_t dv_launch(const float *x, const float *w, const float *bias, float *y, int N, int K,
                          int P, int Q, int C, int R, int S, int H, int W, int stride, int pad,
                          int dil, cudaStream_t st) {
    if (R > kDvMaxTap || S > kDvMaxTap) return CONV2D_ERR_UNSUPPORTED;
    DvParams p;
    p.x = x; p.w = w; p.bias = bias; p.y = y;
    p.N = N; p.K = K; p.P = P; p.Q = Q; p.C = C; p.R = R; p.S = S; p.H = H; p.W = W;
    p.stride = stride; p.pad = pad; p.dil = dil;
    p.tiles_h = (H + kDvRows - 1) / kDvRows;
    p.tiles_w = (W + kDvCols - 1) / kDvCols;
    p.c_blocks = (C + kDvC - 1) / kDvC;
    footprint(stride, dil, R, S, &p.IP, &p.IQ);
    const int64_t grid = (int64_t)N * p.tiles_h * p.tiles_w * p.c_blocks;
    if (grid > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    const size_t bytes = dv_smem_bytes(stride, dil, R, S);
    if (bytes > 96 * 1024) return CONV2D_ERR_UNSUPPORTED;
    if (bytes > 48 * 1024 &&
        cudaFuncSetAttribute(deconv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024) !=
            cudaSuccess)
        return CONV2D_ERR_CUDA;
    deconv_kernel<<<(unsigned)grid, kDvThreads, bytes, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

}  // namespace conv2d
