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
// has at most 256 outputs, else 256 consecutive pixels of one image -- and a
// block of CB output channels (registers; CB = 32, or 8 / 4 for layers with
// that few outputs, such as the decoder's last layer back to the signature
// channels); thread = pixel.  For each chunk of 16 input channels it stages
// the input rows those pixels read (whole rows, zero outside x) and the
// chunk's weights as [k][r][s][CB channels] in shared memory with 4-byte
// asynchronous copies (cp.async, zero-fill outside x), double-buffered: the
// next chunk is in flight while the current one is summed.  Each thread
// keeps bitmasks of its valid filter rows and columns; per valid tap: one input
// read, CB/4 broadcast 16-byte weight reads, CB FFMAs.  (Stride-1 layers with
// few output channels on small images take deconv_s1_kernel, below.)

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kDvThreads = 256;      // = output pixels per CTA (one per thread)
constexpr int kDvK = 16;             // input channels per staged chunk
constexpr int kDvMaxTap = 8;         // R, S <= 8

struct DvParams {
    const float *x, *w, *bias;
    float *y;
    int N, K, P, Q, C, R, S, H, W;
    int stride, pad, dil;
    int imgs;              // > 0: a CTA owns `imgs` whole images (H*W <= 256)
    int tiles_per_img;     // imgs == 0: a CTA owns 256 consecutive pixels of one image
    int tiles, c_blocks;
    int IP, IQ;            // staged input rows per image / columns (= Q)
    uint32_t m_iq, m_ip, m_img;   // reciprocals (sm103a::fdiv) of IQ, IP and kDvK*IP*IQ
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// RT, ST: compile-time filter size bound of the tap loops (kDvMaxTap = any R, S <= 8).
template <int RT, int ST, int CB>
__global__ void __launch_bounds__(kDvThreads, CB <= 8 ? 3 : 2) deconv_kernel(const DvParams p) {
    constexpr int kDvC = CB;
    extern __shared__ float4 dv_smem4[];
    const int nimg = p.imgs > 0 ? p.imgs : 1;
    // two buffers, each [img][kDvK][IP][IQ] inputs then [kDvK][R][S][kDvC] weights
    float *xs = reinterpret_cast<float *>(dv_smem4);
    const int xs_sz = (nimg * kDvK * p.IP * p.IQ + 3) & ~3;
    const int buf_sz = xs_sz + kDvK * p.R * p.S * kDvC;

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

    // Stage input channels [k0, k0 + kDvK) into buffer bf and commit the
    // copies as one group.  Whole images: the chunk of an image,
    // x[n][k0 .. k0+15][..][..], is one contiguous run.  Else the staged rows
    // (channel, input row p_lo + ip) of the CTA's image, zero outside x.
    auto stage = [&](int k0, int bf) {
        const uint32_t xs_u = sm103a::smem_u32(xs + bf * buf_sz);
        const uint32_t ws_u = xs_u + 4u * (uint32_t)xs_sz;
        if (p.imgs > 0) {
            const int per_img = kDvK * plane;              // plane = P*Q here
            const int kn_img = min(kDvK, p.K - k0) * plane;
            for (int i = t; i < nimg * per_img; i += kDvThreads) {
                const int im = sm103a::fdiv(i, p.m_img), f = i - im * per_img;
                const bool in = n0 + im < p.N && f < kn_img;
                sm103a::cp_async_f32(xs_u + 4u * (uint32_t)i,
                                     in ? p.x + ((int64_t)(n0 + im) * p.K + k0) * plane + f : p.x, in);
            }
        } else {
            const int tot = kDvK * plane;
            for (int i = t; i < tot; i += kDvThreads) {
                const int row = sm103a::fdiv(i, p.m_iq), iq = i - row * p.IQ;
                const int kk = sm103a::fdiv(row, p.m_ip), ip = row - kk * p.IP;
                const int k = k0 + kk, pp = p_lo + ip;
                const bool in = k < p.K && (unsigned)pp < (unsigned)p.P;
                sm103a::cp_async_f32(xs_u + 4u * (uint32_t)i,
                                     in ? p.x + (((int64_t)n0 * p.K + k) * p.P + pp) * p.Q + iq : p.x, in);
            }
        }
        // weights: for each input channel the block's w[k][c0 .. c0+CB-1][r][s]
        // are contiguous; read in that order, stored as [k][r*S+s][c]
        const int wrun = kDvC * RS;
        for (int i = t; i < kDvK * wrun; i += kDvThreads) {
            const int kk = i / wrun, f = i - kk * wrun;
            const int j = f / RS, rs = f - j * RS;
            const int k = k0 + kk;
            const bool in = k < p.K && c0 + j < p.C;
            sm103a::cp_async_f32(ws_u + 4u * (uint32_t)((kk * RS + rs) * kDvC + j),
                                 in ? p.w + ((int64_t)k * p.C + c0) * RS + f : p.w, in);
        }
        sm103a::cp_async_commit();
    };

    stage(0, 0);
    int bf = 0;
    for (int k0 = 0; k0 < p.K; k0 += kDvK, bf ^= 1) {
        // every thread is done with the previous chunk, i.e. with the buffer
        // that is refilled here
        __syncthreads();
        if (k0 + kDvK < p.K) {
            stage(k0 + kDvK, bf ^ 1);
            sm103a::cp_async_wait<1>();
        } else {
            sm103a::cp_async_wait<0>();
        }
        __syncthreads();
        const float *ws = xs + bf * buf_sz + xs_sz;
        const int kn = min(kDvK, p.K - k0);
        const float *xi = xs + bf * buf_sz + img * kDvK * plane;
        if constexpr (RT < kDvMaxTap && ST < kDvMaxTap) {
            // Compile-time filter: one staged-input offset per tap and a tap
            // mask, so the loop is branch-free (a warp's pixels can span two
            // output rows with different valid taps): predicated shared read,
            // broadcast weights, CB FFMAs.
            int toff[RT * ST];
            unsigned tmask = 0;
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
                for (int s = 0; s < ST; ++s) {
                    const bool v = ((rmask >> r) & (smask >> s) & 1u) != 0;
                    toff[r * ST + s] = v ? pl[r] * p.IQ + ql[s] : 0;
                    tmask |= (v ? 1u : 0u) << (r * ST + s);
                }
            for (int kk = 0; kk < kn; ++kk) {
                const float *xk = xi + kk * plane;
                const float4 *wk4 = reinterpret_cast<const float4 *>(ws + kk * RT * ST * kDvC);
#pragma unroll
                for (int tp = 0; tp < RT * ST; ++tp) {
                    const float a = ((tmask >> tp) & 1u) ? xk[toff[tp]] : 0.f;
#pragma unroll
                    for (int j = 0; j < kDvC / 4; ++j) {
                        const float4 v = wk4[tp * (kDvC / 4) + j];
                        acc[4 * j] = fmaf(a, v.x, acc[4 * j]);
                        acc[4 * j + 1] = fmaf(a, v.y, acc[4 * j + 1]);
                        acc[4 * j + 2] = fmaf(a, v.z, acc[4 * j + 2]);
                        acc[4 * j + 3] = fmaf(a, v.w, acc[4 * j + 3]);
                    }
                }
            }
            continue;
        }
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

// Stride-1, dilation-1 layers with few output channels on small images
// (the decoder's last layer, back to the signature channels): a CTA owns one
// whole image; thread = 4 consecutive output pixels of a row x CB channels.
// The chunk of kDvS1K input channels of the image is one contiguous run of
// x, staged flat with cp.async (double-buffered), weights as in the gather
// kernel.  Output (h, w) takes input (h + pad - r, w + pad - s): per filter
// row a thread reads the 4 + ST - 1 inputs its pixels share once, then runs
// ST taps x 4 pixels x CB channels of FFMAs on registers.
constexpr int kDvS1K = 8;     // input channels per staged chunk
constexpr int kDvS1Px = 4;    // consecutive output pixels per thread

template <int RT, int ST, int CB>
__global__ void __launch_bounds__(kDvThreads, 3) deconv_s1_kernel(const DvParams p) {
    extern __shared__ float4 dv_smem4[];
    float *sm = reinterpret_cast<float *>(dv_smem4);
    const int plane = p.P * p.Q;
    const int xs_sz = (kDvS1K * plane + 3) & ~3;
    const int buf_sz = xs_sz + kDvS1K * RT * ST * CB;
    sm103a::pdl_wait();
    const int n = blockIdx.x / p.c_blocks;
    const int c0 = (blockIdx.x - n * p.c_blocks) * CB;
    const int t = threadIdx.x;
    const int segs = (p.W + kDvS1Px - 1) / kDvS1Px;
    const int h = t / segs, w0 = (t - h * segs) * kDvS1Px;
    const bool active = h < p.H;
    const int base = w0 + p.pad - (ST - 1);   // input column of register m = base + m

    auto stage = [&](int k0, int bf) {
        const uint32_t xs_u = sm103a::smem_u32(sm + bf * buf_sz);
        const uint32_t ws_u = xs_u + 4u * (uint32_t)xs_sz;
        const int kn = min(kDvS1K, p.K - k0) * plane;
        const float *src = p.x + ((int64_t)n * p.K + k0) * plane;
        for (int i = t; i < kDvS1K * plane; i += kDvThreads)
            sm103a::cp_async_f32(xs_u + 4u * (uint32_t)i, i < kn ? src + i : p.x, i < kn);
        constexpr int wrun = CB * RT * ST;
        for (int i = t; i < kDvS1K * wrun; i += kDvThreads) {
            const int kk = i / wrun, f = i - kk * wrun;
            const int j = f / (RT * ST), rs = f - j * (RT * ST);
            const int k = k0 + kk;
            const bool in = k < p.K && c0 + j < p.C;
            sm103a::cp_async_f32(ws_u + 4u * (uint32_t)((kk * RT * ST + rs) * CB + j),
                                 in ? p.w + ((int64_t)k * p.C + c0) * (RT * ST) + f : p.w, in);
        }
        sm103a::cp_async_commit();
    };

    // channel pairs (2i, 2i + 1) of pixel j, packed for fma.rn.f32x2 (two
    // fp32 FMAs, each rounded as fmaf, per instruction)
    uint64_t acc2[kDvS1Px][CB / 2];
#pragma unroll
    for (int j = 0; j < kDvS1Px; ++j)
#pragma unroll
        for (int i = 0; i < CB / 2; ++i) acc2[j][i] = 0ull;

    stage(0, 0);
    int bf = 0;
    for (int k0 = 0; k0 < p.K; k0 += kDvS1K, bf ^= 1) {
        __syncthreads();                       // every thread is done with the buffer refilled here
        if (k0 + kDvS1K < p.K) {
            stage(k0 + kDvS1K, bf ^ 1);
            sm103a::cp_async_wait<1>();
        } else {
            sm103a::cp_async_wait<0>();
        }
        __syncthreads();
        const float *xs = sm + bf * buf_sz;
        const float4 *ws4 = reinterpret_cast<const float4 *>(xs + xs_sz);
        const int kn = min(kDvS1K, p.K - k0);
        for (int kk = 0; kk < kn; ++kk) {
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                const int ih = h + p.pad - r;
                const bool rv = active && (unsigned)ih < (unsigned)p.P;
                const float *xr = xs + (kk * p.P + (rv ? ih : 0)) * p.Q;
                uint64_t xv2[kDvS1Px + ST - 1];   // each input value twice
#pragma unroll
                for (int m = 0; m < kDvS1Px + ST - 1; ++m) {
                    const int col = base + m;
                    const float v = (rv && (unsigned)col < (unsigned)p.Q) ? xr[col] : 0.f;
                    xv2[m] = sm103a::pack_f32x2(v, v);
                }
#pragma unroll
                for (int s = 0; s < ST; ++s) {
#pragma unroll
                    for (int q = 0; q < CB / 4; ++q) {
                        const float4 wv = ws4[(kk * RT * ST + r * ST + s) * (CB / 4) + q];
                        const uint64_t w01 = sm103a::pack_f32x2(wv.x, wv.y);
                        const uint64_t w23 = sm103a::pack_f32x2(wv.z, wv.w);
#pragma unroll
                        for (int j = 0; j < kDvS1Px; ++j) {
                            const uint64_t a2 = xv2[ST - 1 - s + j];
                            acc2[j][2 * q] = sm103a::ffma2(a2, w01, acc2[j][2 * q]);
                            acc2[j][2 * q + 1] = sm103a::ffma2(a2, w23, acc2[j][2 * q + 1]);
                        }
                    }
                }
            }
        }
    }
    if (!active) return;
    float acc[kDvS1Px][CB];
#pragma unroll
    for (int j = 0; j < kDvS1Px; ++j)
#pragma unroll
        for (int i = 0; i < CB / 2; ++i) sm103a::unpack_f32x2(acc2[j][i], acc[j][2 * i], acc[j][2 * i + 1]);
    float bv[CB];                               // all bias loads before the first store
#pragma unroll
    for (int c = 0; c < CB; ++c) {
        const bool in = p.bias != nullptr && c0 + c < p.C;
        bv[c] = sm103a::ldg_or_zero(in ? p.bias + c0 + c : p.x, in);
    }
    const int64_t HW = (int64_t)p.H * p.W;
    float *yp = p.y + ((int64_t)n * p.C + c0) * HW + (int64_t)h * p.W + w0;
#pragma unroll
    for (int c = 0; c < CB; ++c) {
        if (c0 + c >= p.C) break;
#pragma unroll
        for (int j = 0; j < kDvS1Px; ++j)
            if (w0 + j < p.W) yp[(int64_t)c * HW + j] = acc[j][c] + bv[c];
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

// output channels per CTA: the smallest block that holds C, at most 32
int dv_cblock(int C) { return C <= 4 ? 4 : C <= 8 ? 8 : 32; }

size_t dv_smem_bytes(int H, int W, int P, int Q, int C, int R, int S, int stride, int dil) {
    const int imgs = H * W <= kDvThreads ? std::max(1, kDvThreads / (H * W)) : 1;
    const int ip = stage_rows(H, W, P, R, stride, dil);
    const size_t xs = ((size_t)imgs * kDvK * ip * Q + 3) & ~(size_t)3;
    return 2 * (xs + (size_t)kDvK * R * S * dv_cblock(C)) * sizeof(float);   // two buffers
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
    const int cbk = dv_cblock(C);
    p.c_blocks = (C + cbk - 1) / cbk;
    // stride 1, dilation 1, 2x2 or 3x3, at most 8 output channels, one image
    // per CTA: the register-blocked kernel
    const int64_t s1_bytes = 2 * ((((int64_t)kDvS1K * P * Q + 3) & ~(int64_t)3) + (int64_t)kDvS1K * R * S * cbk) * 4;
    if (stride == 1 && dil == 1 && ((R == 3 && S == 3) || (R == 2 && S == 2)) && C <= 8 &&
        (int64_t)H * ((W + kDvS1Px - 1) / kDvS1Px) <= kDvThreads && s1_bytes <= 96 * 1024 &&
        (int64_t)N * p.c_blocks <= INT32_MAX) {
        void (*k1)(DvParams);
        if (R == 3) k1 = cbk == 4 ? deconv_s1_kernel<3, 3, 4> : deconv_s1_kernel<3, 3, 8>;
        else k1 = cbk == 4 ? deconv_s1_kernel<2, 2, 4> : deconv_s1_kernel<2, 2, 8>;
        if (s1_bytes > 48 * 1024 &&
            cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024) != cudaSuccess)
            return CONV2D_ERR_CUDA;
        if (launch_pdl(k1, dim3((unsigned)(N * p.c_blocks)), dim3(kDvThreads), (size_t)s1_bytes, st, p) !=
            cudaSuccess) {
            cudaGetLastError();
            return CONV2D_ERR_CUDA;
        }
        return CONV2D_OK;
    }
    p.IP = stage_rows(H, W, P, R, stride, dil);
    p.IQ = Q;
    p.m_iq = recip_u32(p.IQ);
    p.m_ip = recip_u32(p.IP);
    p.m_img = recip_u32(kDvK * p.IP * p.IQ);
    const int64_t grid = (int64_t)p.tiles * p.c_blocks;
    if (grid > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    const size_t bytes = dv_smem_bytes(H, W, P, Q, C, R, S, stride, dil);
    if (bytes > 96 * 1024) return CONV2D_ERR_UNSUPPORTED;
    void (*kern)(DvParams);
    auto pick = [&](auto cb) {
        constexpr int B = decltype(cb)::value;
        if (R == 2 && S == 2) kern = deconv_kernel<2, 2, B>;
        else if (R == 3 && S == 3) kern = deconv_kernel<3, 3, B>;
        else kern = deconv_kernel<kDvMaxTap, kDvMaxTap, B>;
    };
    if (cbk == 4) pick(std::integral_constant<int, 4>{});
    else if (cbk == 8) pick(std::integral_constant<int, 8>{});
    else pick(std::integral_constant<int, 32>{});
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
