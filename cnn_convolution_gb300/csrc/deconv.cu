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
// A CTA of 256 threads owns 256 output pixels -- whole images when an image
// has at most 256 outputs, else 256 consecutive pixels of one image -- and
// 32 output channels (registers); thread = pixel.  For each chunk of 16 input
// channels it stages the input rows those pixels read (whole rows, zero
// outside x) and the chunk's weights as [k][r][s][32 channels] in shared
// memory, every staging load issued before the stores.  Each thread keeps
// bitmasks of its valid filter rows and columns; per valid tap: one input
// read, 8 broadcast 16-byte weight reads, 32 FFMAs.

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kDvThreads = 256;      // = output pixels per CTA (one per thread)
constexpr int kDvC = 32;             // output channels per CTA
constexpr int kDvK = 16;             // input channels per staged chunk
constexpr int kDvMaxTap = 8;         // R, S <= 8
constexpr int kDvBatch = 8;          // staging loads in flight per thread

struct DvParams {
    const float *x, *w, *bias;
    float *y;
    int N, K, P, Q, C, R, S, H, W;
    int stride, pad, dil;
    int imgs;              // > 0: a CTA owns `imgs` whole images (H*W <= 256)
    int tiles_per_img;     // imgs == 0: a CTA owns 256 consecutive pixels of one image
    int tiles, c_blocks;
    int IP, IQ;            // staged input rows per image / columns (= Q)
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// RT, ST: compile-time filter size bound of the tap loops (kDvMaxTap = any R, S <= 8).
template <int RT, int ST>
__global__ void __launch_bounds__(kDvThreads, 2) deconv_kernel(const DvParams p) {
    extern __shared__ float4 dv_smem4[];
    const int nimg = p.imgs > 0 ? p.imgs : 1;
    float *xs = reinterpret_cast<float *>(dv_smem4);                   // [img][kDvK][IP][IQ]
    const int xs_sz = (nimg * kDvK * p.IP * p.IQ + 3) & ~3;
    float *ws = xs + xs_sz;                                             // [kDvK][R][S][kDvC]

    // no early trigger: a kernel of many short CTAs lets the next one launch
    // at its exit, so the next grid is spread over idle SMs
    sm103a::pdl_wait();                        // the previous kernel's writes are visible
    const int cb = blockIdx.x % p.c_blocks;
    const int tile = blockIdx.x / p.c_blocks;
    const int c0 = cb * kDvC;
    const int HW = p.H * p.W;
    // this CTA's images and pixels
    int n0, pix0, p_lo;
    if (p.imgs > 0) {
        n0 = tile * p.imgs;
        pix0 = 0;
        p_lo = 0;
    } else {
        n0 = tile / p.tiles_per_img;
        pix0 = (tile - n0 * p.tiles_per_img) * kDvThreads;
        const int h_first = pix0 / p.W;
        p_lo = floor_div(h_first + p.pad - (p.R - 1) * p.dil + p.stride - 1, p.stride);
    }
    const int t = threadIdx.x;
    const int img = p.imgs > 0 ? t / HW : 0;
    const int pix = p.imgs > 0 ? t - img * HW : pix0 + t;
    const int n = n0 + img;
    const bool active = n < p.N && pix < HW && (p.imgs == 0 || img < p.imgs);
    const int h = active ? pix / p.W : 0, wcol = active ? pix - h * p.W : 0;

    // valid taps of this pixel, with staged row / column indices
    unsigned rmask = 0, smask = 0;
    int pl[RT], ql[ST];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        pl[r] = 0;
        const int hp = h + p.pad - r * p.dil;
        if (active && r < p.R && hp >= 0 && hp % p.stride == 0 && hp / p.stride < p.P) {
            rmask |= 1u << r;
            pl[r] = hp / p.stride - p_lo;
        }
    }
#pragma unroll
    for (int s = 0; s < ST; ++s) {
        ql[s] = 0;
        const int wp = wcol + p.pad - s * p.dil;
        if (active && s < p.S && wp >= 0 && wp % p.stride == 0 && wp / p.stride < p.Q) {
            smask |= 1u << s;
            ql[s] = wp / p.stride;
        }
    }

    float acc[kDvC];
#pragma unroll
    for (int j = 0; j < kDvC; ++j) acc[j] = 0.f;
    // exact compile-time filter sizes make the staging index arithmetic cheap
    const int RS = (RT < kDvMaxTap && RT * ST > 0) ? RT * ST : p.R * p.S;
    const int plane = p.IP * p.IQ;
    const int warp = t / 32, lane = t % 32;

    for (int k0 = 0; k0 < p.K; k0 += kDvK) {
        __syncthreads();
        // stage x.  Whole images: the chunk of an image, x[n][k0 .. k0+15][..][..],
        // is one contiguous run, copied flat.  Else one staged row (image,
        // channel, input row) per warp pass, lanes along the row; 4 rows in
        // flight per warp.
        const int nrows = p.imgs > 0 ? 0 : nimg * kDvK * p.IP;
        if (p.imgs > 0) {
            const int per_img = kDvK * plane;              // plane = P*Q here
            const int kn_img = min(kDvK, p.K - k0) * plane;
            for (int i0 = 0; i0 < nimg * per_img; i0 += kDvThreads * kDvBatch) {
                float v[kDvBatch];
#pragma unroll
                for (int u = 0; u < kDvBatch; ++u) {
                    const int i = i0 + u * kDvThreads + t;
                    const int im = i / per_img, f = i - im * per_img;
                    const bool in = i < nimg * per_img && n0 + im < p.N && f < kn_img;
                    v[u] = sm103a::ldg_or_zero(in ? p.x + ((int64_t)(n0 + im) * p.K + k0) * plane + f : p.x, in);
                }
#pragma unroll
                for (int u = 0; u < kDvBatch; ++u) {
                    const int i = i0 + u * kDvThreads + t;
                    if (i < nimg * per_img) xs[i] = v[u];
                }
            }
        }
        for (int row0 = warp * 4; row0 < nrows; row0 += (kDvThreads / 32) * 4) {
            float v[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int row = row0 + u;
                const int ip = row % p.IP, r2 = row / p.IP;
                const int kk = r2 % kDvK, im = r2 / kDvK;
                const int k = k0 + kk, pp = p_lo + ip, nn = n0 + im;
                const bool rin = row < nrows && nn < p.N && k < p.K && (unsigned)pp < (unsigned)p.P;
                const float *src = p.x + (((int64_t)nn * p.K + k) * p.P + pp) * p.Q;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int iq = lane + 32 * e;
                    const bool in = rin && iq < p.Q;
                    v[u][e] = sm103a::ldg_or_zero(in ? src + iq : p.x, in);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int row = row0 + u;
                if (row < nrows) {
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (lane + 32 * e < p.IQ) xs[row * p.IQ + lane + 32 * e] = v[u][e];
                }
            }
            // rows longer than 64 columns (wide outputs): the rest, plainly
            for (int u = 0; u < 4 && p.IQ > 64; ++u) {
                const int row = row0 + u;
                if (row >= nrows) break;
                const int ip = row % p.IP, r2 = row / p.IP;
                const int kk = r2 % kDvK, im = r2 / kDvK;
                const int k = k0 + kk, pp = p_lo + ip, nn = n0 + im;
                const bool rin = nn < p.N && k < p.K && (unsigned)pp < (unsigned)p.P;
                for (int iq = 64 + lane; iq < p.IQ; iq += 32)
                    xs[row * p.IQ + iq] = rin ? __ldg(p.x + (((int64_t)nn * p.K + k) * p.P + pp) * p.Q + iq) : 0.f;
            }
        }
        // stage w: for each input channel the block's weights w[k][c0 .. c0+31][r][s]
        // are contiguous; read them in that order, store as [k][r*S+s][c]
        const int wrun = kDvC * RS;
        for (int i0 = 0; i0 < kDvK * wrun; i0 += kDvThreads * kDvBatch) {
            float v[kDvBatch];
#pragma unroll
            for (int u = 0; u < kDvBatch; ++u) {
                const int i = i0 + u * kDvThreads + t;
                const int kk = i / wrun, f = i - kk * wrun;
                const int k = k0 + kk, c = c0 + f / RS;
                const bool in = i < kDvK * wrun && k < p.K && c < p.C;
                v[u] = sm103a::ldg_or_zero(in ? p.w + ((int64_t)k * p.C + c0) * RS + f : p.w, in);
            }
#pragma unroll
            for (int u = 0; u < kDvBatch; ++u) {
                const int i = i0 + u * kDvThreads + t;
                if (i < kDvK * wrun) {
                    const int kk = i / wrun, f = i - kk * wrun;
                    const int j = f / RS, rs = f - j * RS;
                    ws[(kk * RS + rs) * kDvC + j] = v[u];
                }
            }
        }
        __syncthreads();
        const int kn = min(kDvK, p.K - k0);
        const float *xi = xs + img * kDvK * plane;
        for (int kk = 0; kk < kn; ++kk) {
            const float *xk = xi + kk * plane;
            const float *wk = ws + kk * RS * kDvC;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                if (!((rmask >> r) & 1u)) continue;
                const float *xr = xk + pl[r] * p.IQ;
#pragma unroll
                for (int s = 0; s < ST; ++s) {
                    if (!((smask >> s) & 1u)) continue;
                    const float a = xr[ql[s]];
                    const float4 *w4 = reinterpret_cast<const float4 *>(wk + (r * (ST < kDvMaxTap ? ST : p.S) + s) * kDvC);
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
    if (!active) return;
    if (p.bias) {                              // all bias loads before the first store
        float bv[kDvC];
#pragma unroll
        for (int j = 0; j < kDvC; ++j) bv[j] = sm103a::ldg_or_zero(p.bias + (c0 + j < p.C ? c0 + j : 0), c0 + j < p.C);
#pragma unroll
        for (int j = 0; j < kDvC; ++j) acc[j] += bv[j];
    }
    float *yp = p.y + ((int64_t)n * p.C + c0) * HW + pix;
#pragma unroll
    for (int j = 0; j < kDvC; ++j) {
        if (c0 + j < p.C) yp[(int64_t)j * HW] = acc[j];
    }
}

// Staged input rows per image for a CTA's pixels (an upper bound).
int stage_rows(int H, int W, int P, int R, int stride, int dil) {
    if (H * W <= kDvThreads) return P;
    // rows p_lo .. p_lo + IP - 1 are staged (zero outside [0, P)); p_lo may be
    // negative, so the count is not clamped to P
    const int rows_out = (kDvThreads + W - 1) / W + 1;            // output rows 256 pixels can touch
    return (rows_out - 1 + (R - 1) * dil) / stride + 2;
}

}  // namespace

size_t dv_smem_bytes(int H, int W, int P, int Q, int R, int S, int stride, int dil) {
    const int imgs = H * W <= kDvThreads ? std::max(1, kDvThreads / (H * W)) : 1;
    const int ip = stage_rows(H, W, P, R, stride, dil);
    const size_t xs = ((size_t)imgs * kDvK * ip * Q + 3) & ~(size_t)3;
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
    const int64_t HW = (int64_t)H * W;
    if (HW <= kDvThreads) {
        p.imgs = (int)std::max<int64_t>(1, kDvThreads / HW);
        p.tiles_per_img = 0;
        p.tiles = (int)((N + p.imgs - 1) / p.imgs);
    } else {
        p.imgs = 0;
        p.tiles_per_img = (int)((HW + kDvThreads - 1) / kDvThreads);
        const int64_t tiles = (int64_t)N * p.tiles_per_img;
        if (tiles > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
        p.tiles = (int)tiles;
    }
    p.c_blocks = (C + kDvC - 1) / kDvC;
    p.IP = stage_rows(H, W, P, R, stride, dil);
    p.IQ = Q;
    const int64_t grid = (int64_t)p.tiles * p.c_blocks;
    if (grid > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    const size_t bytes = dv_smem_bytes(H, W, P, Q, R, S, stride, dil);
    if (bytes > 96 * 1024) return CONV2D_ERR_UNSUPPORTED;
    void (*kern)(DvParams);
    if (R == 2 && S == 2) kern = deconv_kernel<2, 2>;
    else if (R == 3 && S == 3) kern = deconv_kernel<3, 3>;
    else kern = deconv_kernel<kDvMaxTap, kDvMaxTap>;
    if (bytes > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    if (launch_pdl(kern, dim3((unsigned)grid), dim3(kDvThreads), bytes, st, p) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

}  // namespace conv2d
