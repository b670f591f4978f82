// Direct fp32 convolution for layers with a short reduction (C*R*S <= 64),
// such as the first MSCRED encoder layer (3 signature-matrix channels, 3x3).
//
// The plain definition of the forward convolution as "GPU-Accelerating
// MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch Extension" states it
// (section "Understanding the Convolution Operation": every output is the
// bias plus the sum over input channels and filter taps of input x weight),
// computed without any lowering: with only C*R*S <= 64 products per output
// the im2col / GEMM machinery costs more than the arithmetic.
//
// A CTA of 128 threads owns an 8 x 32 block of output pixels of one image
// and every output channel; four CTAs share an SM (small blocks keep the
// most loaded SM close to the average when the blocks do not divide evenly
// over the SMs).  It stages the zero-padded input patch that
// block reads ([C][IH][IW]) and the weights transposed to [C*R*S][K] in
// shared memory, then each thread accumulates 2 pixels (rows 2w, 2w+1 of the
// block, column = lane) x 32 channels in registers: per filter tap, 2 patch
// reads and 8 broadcast 16-byte weight reads feed 64 FFMAs.  Channel blocks
// of 32 repeat over the same staged patch.  (A 16-channel block at 64
// registers per thread measured slower on GB300: the cap forces spills.)
// Zero padding lives in the patch, so the inner loop has no bounds tests.  NCHW stores are coalesced across
// the lanes of a warp (consecutive q); NHWC stores are 16-byte vectors.

#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

constexpr int kDcThreads = 128;
constexpr int kDcRows = 8;       // output rows per CTA (2 per warp)
constexpr int kDcCols = 32;      // output columns per CTA (1 per lane)
constexpr int kDcKc = 32;        // output channels per register block

struct DcParams {
    const float *x, *w, *bias;
    float *y;
    int N, C, H, W, K, R, S, P, Q;
    int stride, pad, dil;
    int IH, IW;           // staged patch rows / columns
    int Kp;               // K rounded up to kDcKc (row length of the transposed weights)
    int tiles_p, tiles_q;
    int nhwc;
    // reciprocals for the staging index arithmetic (sm103a::fdiv): IW, IH, Kp, R*S
    uint32_t m_iw, m_ih, m_kp, m_rs;
};

// The staged patch and weight table are bounded by the shared-memory limit,
// so every index and divisor given to sm103a::fdiv meets its n * d < 2^32.
using sm103a::fdiv;

// RT, ST: compile-time filter size (0 = read from the parameters).
template <int RT, int ST>
__global__ void __launch_bounds__(kDcThreads, 4) direct_conv_kernel(const DcParams p) {
    extern __shared__ float4 dc_smem4[];
    const int R = RT > 0 ? RT : p.R;
    const int S = ST > 0 ? ST : p.S;
    float *xs = reinterpret_cast<float *>(dc_smem4);           // [C][IH][IW]
    const int plane = p.IH * p.IW;
    const int patch = p.C * plane;
    const int RS = R * S;
    const int Kg = p.C * RS;
    float *wt = xs + ((patch + 3) & ~3);                       // [Kg][Kp], 16-byte aligned rows

    int t = blockIdx.x;
    const int tq = t % p.tiles_q;
    t /= p.tiles_q;
    const int tp = t % p.tiles_p;
    const int n = t / p.tiles_p;
    const int p0 = tp * kDcRows, q0 = tq * kDcCols;
    const int h0 = p0 * p.stride - p.pad, w0 = q0 * p.stride - p.pad;
    sm103a::pdl_launch_dependents();
    sm103a::pdl_wait();                        // the previous kernel's writes are visible

    // Stage the input patch (zero outside the image) and the weights as
    // [g = (c, r, s)][k] (zero for k >= K) with 4-byte asynchronous copies
    // (cp.async; a copy outside the image writes zero): every copy of the
    // CTA is in flight at once, and no register holds them.
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float *ximg = p.x + (int64_t)n * p.C * p.H * p.W;   // this image (C*H*W < 2^31)
    const uint32_t xs_u = sm103a::smem_u32(xs), wt_u = sm103a::smem_u32(wt);
    for (int i = (int)threadIdx.x; i < patch; i += kDcThreads) {
        const int r2 = fdiv(i, p.m_iw);
        const int iw = i - r2 * p.IW;
        const int c = fdiv(r2, p.m_ih);
        const int ih = r2 - c * p.IH;
        const int h = h0 + ih, wc = w0 + iw;
        const bool in = (unsigned)h < (unsigned)p.H && (unsigned)wc < (unsigned)p.W;
        const int hh = in ? h : 0, ww = in ? wc : 0, cc = in ? c : 0;   // in-image: no overflow
        const int off = p.nhwc ? (hh * p.W + ww) * p.C + cc : (cc * p.H + hh) * p.W + ww;
        sm103a::cp_async_f32(xs_u + 4u * (uint32_t)i, ximg + off, in);
    }
    const int wn = Kg * p.Kp;
    for (int i = (int)threadIdx.x; i < wn; i += kDcThreads) {
        const int g = fdiv(i, p.m_kp), k = i - g * p.Kp;
        int woff = g;                       // offset of w[k = 0][g]
        if (p.nhwc) {
            const int c = fdiv(g, p.m_rs), rs = g - c * RS;
            woff = rs * p.C + c;
        }
        const bool in = k < p.K;
        sm103a::cp_async_f32(wt_u + 4u * (uint32_t)i, p.w + (in ? (int64_t)k * Kg + woff : 0), in);
    }
    sm103a::cp_async_commit();
    sm103a::cp_async_wait<0>();
    __syncthreads();

    const int pr0 = 2 * warp;                      // this thread's first row in the block
    const int pa = p0 + pr0, pb = pa + 1, q = q0 + lane;
    const bool va = pa < p.P && q < p.Q, vb = pb < p.P && q < p.Q;
    const int xa = (pr0 * p.stride) * p.IW + lane * p.stride;
    const int xb = xa + p.stride * p.IW;
    const int64_t PQ = (int64_t)p.P * p.Q;

    for (int kc = 0; kc < p.K; kc += kDcKc) {
        float acc_a[kDcKc], acc_b[kDcKc];
#pragma unroll
        for (int j = 0; j < kDcKc; ++j) acc_a[j] = acc_b[j] = 0.f;
        const float *wrow = wt + kc;
        for (int c = 0; c < p.C; ++c) {
            const float *xc = xs + c * plane;
#pragma unroll
            for (int r = 0; r < (RT > 0 ? RT : 1); ++r) {
                for (int rr = (RT > 0 ? r : 0); rr < (RT > 0 ? r + 1 : R); ++rr) {
                    const float *xr = xc + rr * p.dil * p.IW;
#pragma unroll
                    for (int s0 = 0; s0 < (ST > 0 ? ST : 1); ++s0) {
                        for (int ss = (ST > 0 ? s0 : 0); ss < (ST > 0 ? s0 + 1 : S); ++ss) {
                            const float a = xr[xa + ss * p.dil];
                            const float b = xr[xb + ss * p.dil];
                            const float4 *w4 = reinterpret_cast<const float4 *>(wrow);
#pragma unroll
                            for (int j = 0; j < kDcKc / 4; ++j) {
                                const float4 wv = w4[j];
                                acc_a[4 * j] = fmaf(a, wv.x, acc_a[4 * j]);
                                acc_a[4 * j + 1] = fmaf(a, wv.y, acc_a[4 * j + 1]);
                                acc_a[4 * j + 2] = fmaf(a, wv.z, acc_a[4 * j + 2]);
                                acc_a[4 * j + 3] = fmaf(a, wv.w, acc_a[4 * j + 3]);
                                acc_b[4 * j] = fmaf(b, wv.x, acc_b[4 * j]);
                                acc_b[4 * j + 1] = fmaf(b, wv.y, acc_b[4 * j + 1]);
                                acc_b[4 * j + 2] = fmaf(b, wv.z, acc_b[4 * j + 2]);
                                acc_b[4 * j + 3] = fmaf(b, wv.w, acc_b[4 * j + 3]);
                            }
                            wrow += p.Kp;
                        }
                    }
                }
            }
        }
        // + bias (all loads before the first store), store
        const int kn = min(kDcKc, p.K - kc);
        if (p.bias) {
            float bv[kDcKc];
#pragma unroll
            for (int j = 0; j < kDcKc; ++j) bv[j] = sm103a::ldg_or_zero(p.bias + (j < kn ? kc + j : 0), j < kn);
#pragma unroll
            for (int j = 0; j < kDcKc; ++j) {
                acc_a[j] += bv[j];
                acc_b[j] += bv[j];
            }
        }
        if (p.nhwc) {
            float *ya = p.y + (((int64_t)n * p.P + pa) * p.Q + q) * p.K + kc;
            float *yb = ya + (int64_t)p.Q * p.K;
            const bool vec = (p.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.y) & 15) == 0);
#pragma unroll
            for (int j = 0; j < kDcKc; j += 4) {
                if (j >= kn) break;
                if (vec) {
                    if (va) *reinterpret_cast<float4 *>(ya + j) =
                        make_float4(acc_a[j], acc_a[j + 1], acc_a[j + 2], acc_a[j + 3]);
                    if (vb) *reinterpret_cast<float4 *>(yb + j) =
                        make_float4(acc_b[j], acc_b[j + 1], acc_b[j + 2], acc_b[j + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (j + e < kn) {
                            if (va) ya[j + e] = acc_a[j + e];
                            if (vb) yb[j + e] = acc_b[j + e];
                        }
                    }
                }
            }
        } else {
            float *ya = p.y + ((int64_t)n * p.K + kc) * PQ + (int64_t)pa * p.Q + q;
            float *yb = ya + p.Q;
#pragma unroll
            for (int j = 0; j < kDcKc; ++j) {
                if (j < kn) {
                    if (va) ya[(int64_t)j * PQ] = acc_a[j];
                    if (vb) yb[(int64_t)j * PQ] = acc_b[j];
                }
            }
        }
    }
}

// ------------------------------------------------------------------ quad kernel
//
// Register-blocked variant for stride-1, dilation-1 layers with at most 32
// output channels and 1x1, 3x3 or 5x5 filters (the MSCRED encoder's first
// layer and the single signature-matrix convolution).  Same CTA block and
// staging as above (8 x 32 output pixels, 128 threads), but a thread owns 4
// consecutive output pixels of one row x 16 output channels.  Per (input
// channel, filter row) it reads the 8 patch values its pixels' S taps share
// with two 16-byte shared loads and runs S taps x 4 pixels x 16 channels of
// FFMAs from registers, reading each tap's 16 weights as four 16-byte
// broadcasts: 2 + 4S shared loads per 64S FFMAs (the kernel above issues 10
// per 64).  The FMAs run as packed fma.rn.f32x2 on channel pairs (the pixel
// value duplicated, two weights, two accumulators): the same FMA rate in
// half the issue slots, which took the MSCRED layer from 22.5 to 18.0 us.
// Patch rows are padded to kQdIWP = 36 floats so the 16-byte loads stay
// aligned.
constexpr int kQdIWP = 36;

template <int R, int S>
__global__ void __launch_bounds__(kDcThreads, 4) direct_quad_kernel(const DcParams p) {
    extern __shared__ float4 dc_smem4[];
    constexpr int IH = kDcRows + R - 1;
    constexpr int plane = IH * kQdIWP;
    float *xs = reinterpret_cast<float *>(dc_smem4);           // [C][IH][kQdIWP]
    const int patch = p.C * plane;                             // a multiple of 4
    const int Kg = p.C * R * S;
    float *wt = xs + patch;                                    // [Kg][32]

    int t = blockIdx.x;
    const int tq = t % p.tiles_q;
    t /= p.tiles_q;
    const int tp = t % p.tiles_p;
    const int n = t / p.tiles_p;
    const int p0 = tp * kDcRows, q0 = tq * kDcCols;
    const int h0 = p0 - p.pad, w0 = q0 - p.pad;
    sm103a::pdl_launch_dependents();
    sm103a::pdl_wait();

    const float *ximg = p.x + (int64_t)n * p.C * p.H * p.W;
    const uint32_t xs_u = sm103a::smem_u32(xs), wt_u = sm103a::smem_u32(wt);
    for (int i = (int)threadIdx.x; i < patch; i += kDcThreads) {
        const int r2 = fdiv(i, p.m_iw);
        const int iw = i - r2 * kQdIWP;
        const int c = fdiv(r2, p.m_ih);
        const int ih = r2 - c * IH;
        const int h = h0 + ih, wc = w0 + iw;
        const bool in = (unsigned)h < (unsigned)p.H && (unsigned)wc < (unsigned)p.W;
        const int hh = in ? h : 0, ww = in ? wc : 0, cc = in ? c : 0;
        const int off = p.nhwc ? (hh * p.W + ww) * p.C + cc : (cc * p.H + hh) * p.W + ww;
        sm103a::cp_async_f32(xs_u + 4u * (uint32_t)i, ximg + off, in);
    }
    for (int i = (int)threadIdx.x; i < Kg * 32; i += kDcThreads) {
        const int g = i >> 5, k = i & 31;
        int woff = g;
        if (p.nhwc) {
            const int c = fdiv(g, p.m_rs), rs = g - c * (R * S);
            woff = rs * p.C + c;
        }
        const bool in = k < p.K;
        sm103a::cp_async_f32(wt_u + 4u * (uint32_t)i, p.w + (in ? (int64_t)k * Kg + woff : 0), in);
    }
    sm103a::cp_async_commit();
    sm103a::cp_async_wait<0>();
    __syncthreads();

    // warps 0-1: channels 0-15, warps 2-3: 16-31; a warp = 8 quads x 4 rows
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int kb = warp >> 1;
    const int rho = (warp & 1) * 4 + (lane >> 3);
    const int j = lane & 7;
    uint64_t acc2[4][8];                       // channel pairs (2kk, 2kk + 1) of pixel a
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) acc2[a][kk] = 0ull;
    const float *xt = xs + rho * kQdIWP + 4 * j;
    const float *wk = wt + kb * 16;
    for (int c = 0; c < p.C; ++c) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 v0 = *reinterpret_cast<const float4 *>(xt + (c * IH + r) * kQdIWP);
            const float4 v1 = *reinterpret_cast<const float4 *>(xt + (c * IH + r) * kQdIWP + 4);
            const float xv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int s2 = 0; s2 < S; ++s2) {
                const float4 *w4 = reinterpret_cast<const float4 *>(wk + ((c * R + r) * S + s2) * 32);
                uint64_t w2[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 t4 = w4[q];
                    w2[2 * q] = sm103a::pack_f32x2(t4.x, t4.y);
                    w2[2 * q + 1] = sm103a::pack_f32x2(t4.z, t4.w);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const uint64_t xx = sm103a::pack_f32x2(xv[a + s2], xv[a + s2]);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) acc2[a][kk] = sm103a::ffma2(xx, w2[kk], acc2[a][kk]);
                }
            }
        }
    }
    float acc[4][16];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) sm103a::unpack_f32x2(acc2[a][kk], acc[a][2 * kk], acc[a][2 * kk + 1]);
    // + bias, store
    const int k0 = kb * 16;
    if (p.bias) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float bv = sm103a::ldg_or_zero(p.bias + (k0 + k < p.K ? k0 + k : 0), k0 + k < p.K);
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a][k] += bv;
        }
    }
    const int pp = p0 + rho;
    if (pp >= p.P) return;
    const int q = q0 + 4 * j;
    if (p.nhwc) {
        const bool vec = (p.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.y) & 15) == 0);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            if (q + a >= p.Q) break;
            float *yr = p.y + (((int64_t)n * p.P + pp) * p.Q + q + a) * p.K + k0;
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                if (k0 + k >= p.K) break;
                if (vec)
                    *reinterpret_cast<float4 *>(yr + k) = make_float4(acc[a][k], acc[a][k + 1], acc[a][k + 2], acc[a][k + 3]);
                else
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k0 + k + e < p.K) yr[k + e] = acc[a][k + e];
            }
        }
    } else {
        const int64_t PQ = (int64_t)p.P * p.Q;
        float *yr = p.y + ((int64_t)n * p.K + k0) * PQ + (int64_t)pp * p.Q + q;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k0 + k >= p.K) break;
#pragma unroll
            for (int a = 0; a < 4; ++a)
                if (q + a < p.Q) yr[(int64_t)k * PQ + a] = acc[a][k];
        }
    }
}

// The quad kernel takes stride-1, dilation-1 layers with K <= 32 and a 1x1,
// 3x3 or 5x5 filter (the patch row of 32 + S - 1 columns fits kQdIWP).
bool quad_ok(const Shape &s) {
    return s.stride == 1 && s.dil == 1 && s.K <= 32 && s.R == s.S && (s.R == 1 || s.R == 3 || s.R == 5);
}

void patch_dims(const Shape &s, int *ih, int *iw) {
    *ih = (kDcRows - 1) * s.stride + (s.R - 1) * s.dil + 1;
    *iw = quad_ok(s) ? kQdIWP : (kDcCols - 1) * s.stride + (s.S - 1) * s.dil + 1;
}

}  // namespace

size_t dc_smem_bytes(const Shape &s) {
    int ih, iw;
    patch_dims(s, &ih, &iw);
    const size_t patch = ((size_t)s.C * ih * iw + 3) & ~(size_t)3;
    const size_t kp = ((size_t)s.K + kDcKc - 1) / kDcKc * kDcKc;   // 32 for the quad kernel
    return (patch + (size_t)s.Kg * kp) * sizeof(float);
}

bool dc_shape_ok(const Shape &s) {
    if (s.dtype != CONV2D_F32) return false;
    if (s.Kg > 64 || s.stride > 4 || (int64_t)s.dil * (s.R - 1) > 64 || (int64_t)s.dil * (s.S - 1) > 64)
        return false;
    if ((int64_t)s.N * ((s.P + kDcRows - 1) / kDcRows) * ((s.Q + kDcCols - 1) / kDcCols) > INT32_MAX)
        return false;
    if ((int64_t)s.C * s.H * s.W >= ((int64_t)1 << 31)) return false;   // 32-bit offsets within an image
    return dc_smem_bytes(s) <= 96 * 1024;
}


void dc_block(int *rows, int *cols, int *threads, int *kc) {
    *rows = kDcRows;
    *cols = kDcCols;
    *threads = kDcThreads;
    *kc = kDcKc;
}

int dc_grid(const Shape &s) {
    return (int)((int64_t)s.N * ((s.P + kDcRows - 1) / kDcRows) * ((s.Q + kDcCols - 1) / kDcCols));
}

conv2d_status_t dc_launch(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    (void)pl;
    DcParams p;
    p.x = static_cast<const float *>(t.x);
    p.w = static_cast<const float *>(t.w);
    p.bias = static_cast<const float *>(t.bias);
    p.y = static_cast<float *>(t.y);
    p.N = s.N; p.C = s.C; p.H = s.H; p.W = s.W; p.K = s.K; p.R = s.R; p.S = s.S;
    p.P = s.P; p.Q = s.Q;
    p.stride = s.stride; p.pad = s.pad; p.dil = s.dil;
    patch_dims(s, &p.IH, &p.IW);
    p.Kp = (s.K + kDcKc - 1) / kDcKc * kDcKc;
    p.tiles_p = (s.P + kDcRows - 1) / kDcRows;
    p.tiles_q = (s.Q + kDcCols - 1) / kDcCols;
    p.nhwc = s.layout == CONV2D_NHWC ? 1 : 0;
    p.m_iw = recip_u32(p.IW);
    p.m_ih = recip_u32(p.IH);
    p.m_kp = recip_u32(p.Kp);
    p.m_rs = recip_u32(s.R * s.S);
    const size_t bytes = dc_smem_bytes(s);
    void (*kern)(DcParams);
    if (quad_ok(s)) {
        if (s.R == 3) kern = direct_quad_kernel<3, 3>;
        else if (s.R == 1) kern = direct_quad_kernel<1, 1>;
        else kern = direct_quad_kernel<5, 5>;
    } else if (s.R == 3 && s.S == 3) kern = direct_conv_kernel<3, 3>;
    else if (s.R == 2 && s.S == 2) kern = direct_conv_kernel<2, 2>;
    else if (s.R == 1 && s.S == 1) kern = direct_conv_kernel<1, 1>;
    else if (s.R == 5 && s.S == 5) kern = direct_conv_kernel<5, 5>;
    else kern = direct_conv_kernel<0, 0>;
    if (bytes > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    if (launch_pdl(kern, dim3(dc_grid(s)), dim3(kDcThreads), bytes, st, p) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

}  // namespace conv2d
