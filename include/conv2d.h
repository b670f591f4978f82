/*
 * conv2d.h -- C ABI of the GB300 forward 2-D convolution library
 *             (libconv2d_gb300.so).
 *
 * The operation (one call = one layer):
 *
 *   y[n,k,p,q] = bias[k] + sum_{c<C, r<R, s<S} x[n, c, p*stride - pad + r*dil,
 *                                                q*stride - pad + s*dil] * w[k,c,r,s]
 *
 * x is read as zero outside 0 <= h < H, 0 <= w < W (zero padding); the
 * filter is not flipped (cross-correlation); and
 *
 *   P = floor((H + 2*pad - dil*(R-1) - 1) / stride) + 1,
 *   Q = floor((W + 2*pad - dil*(S-1) - 1) / stride) + 1.
 *
 * This is the convolution of "GPU-Accelerating MSCRED with CUDA, im2col, GEMM,
 * and a Custom PyTorch Extension" (sections "Where the Performance Bottleneck
 * Appeared" and "Transforming Conv2D into im2col and GEMM": output = weight
 * matrix x im2col(input)) and of "Enabling Memory-efficient Im2win Convolution
 * with Multi-precision Support on GPU CUDA and Tensor Cores" (abstract: full
 * precision on CUDA cores, half precision on tensor cores).  Unlike the
 * im2col formulation, no im2col matrix is ever built: the library needs no
 * workspace at all (conv2d_workspace_bytes reports 0).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, contiguous and caller-owned device memory (cudaMalloc,
 *    cudaMallocAsync or managed memory; torch tensors qualify).  Host pointers
 *    are rejected with CONV2D_ERR_INVALID_ARG before anything is launched.
 *  - dtype applies to x, w, bias and y alike.  CONV2D_F32 results meet the
 *    fp32 bound |y - y_exact| <= 1e-6 * (sum |x||w| + |bias|) on every
 *    kernel.  By default (CONV2D_ALGO_AUTO) the chooser runs an fp32 layer
 *    either on tensor cores as split-precision 3xTF32 (each operand split
 *    into two TF32 parts, three tcgen05 kind::tf32 products per multiply-add,
 *    the full-magnitude term summed per 32-element stage in fp32 registers)
 *    or on CUDA cores (FFMA), whichever its cost model expects to be faster;
 *    plain single-pass TF32 is never used.  CONV2D_ALGO_CUDA_CORE keeps a
 *    layer on FFMA.  CONV2D_F16 / CONV2D_BF16 multiply in the input type and
 *    accumulate in fp32; y is rounded once, to nearest even.
 *  - layout CONV2D_NCHW: x [N][C][H][W], w [K][C][R][S], y [N][K][P][Q].
 *    layout CONV2D_NHWC: x [N][H][W][C], w [K][R][S][C], y [N][P][Q][K].
 *    bias is [K] or NULL (read as zero).
 *  - stride, pad and dil apply to both spatial axes.
 *  - y must not overlap x, w or bias.
 *  - Pointers must be aligned to the element size; the tensor-core path is used
 *    only when x, w, y are 16-byte aligned and C, K are multiples of 8 (other
 *    inputs take the CUDA-core path; they do not fail).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *    allocate nothing.  Errors are returned, never thrown; argument errors are
 *    detected before any launch.  A kernel that gives up waiting on an internal
 *    barrier (it never should) records CONV2D_ERR_TIMEOUT in a device status
 *    word, read by conv2d_get_device_status().
 *  - All entry points are thread-safe.
 */
#ifndef CONV2D_GB300_H
#define CONV2D_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV2D_OK = 0,
    CONV2D_ERR_INVALID_ARG = 1,   /* bad size, null or host pointer, aliasing, empty output */
    CONV2D_ERR_UNSUPPORTED = 2,   /* dtype/layout/algo combination not provided */
    CONV2D_ERR_MISALIGNED = 3,    /* a pointer is not aligned to its element size */
    CONV2D_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch, attribute) */
    CONV2D_ERR_TIMEOUT = 5,       /* a kernel gave up on a bounded barrier wait */
    CONV2D_ERR_INTERNAL = 6
} conv2d_status_t;

typedef enum { CONV2D_F32 = 0, CONV2D_F16 = 1, CONV2D_BF16 = 2 } conv2d_dtype_t;
typedef enum { CONV2D_NCHW = 0, CONV2D_NHWC = 1 } conv2d_layout_t;

/* Kernel family.  AUTO lets the per-shape chooser decide. */
typedef enum {
    CONV2D_ALGO_AUTO = 0,
    CONV2D_ALGO_CUDA_CORE = 1,    /* shared-memory implicit GEMM on FFMA, any dtype/layout */
    CONV2D_ALGO_TENSOR_CORE = 2   /* tcgen05 implicit GEMM: f16/bf16 NHWC (TMA im2col / windows),
                                     or fp32 either layout as split-precision 3xTF32 */
} conv2d_algo_t;

typedef struct conv2d_desc *conv2d_desc_t;

/*
 * Create a layer descriptor (a host object owned by the caller; destroy it
 * with conv2d_desc_destroy).  Validates every size:
 * N,C,H,W,K,R,S,stride,dil >= 1, pad >= 0, P,Q >= 1, element counts below
 * 2^40.  Returns CONV2D_ERR_INVALID_ARG (and leaves *out untouched) otherwise.
 */
conv2d_status_t conv2d_desc_create(conv2d_desc_t *out, int N, int C, int H, int W,
                                   int K, int R, int S, int stride, int pad, int dil,
                                   conv2d_dtype_t dtype, conv2d_layout_t layout);

/* Free a descriptor.  NULL is accepted. */
conv2d_status_t conv2d_desc_destroy(conv2d_desc_t desc);

/* Output spatial extents P, Q of the descriptor's layer. */
conv2d_status_t conv2d_output_dims(conv2d_desc_t desc, int *P, int *Q);

/*
 * Device memory a forward call needs beyond x, w, bias and y.  Always 0: the
 * windows of x are staged straight from x into shared memory, never into a
 * materialised im2col matrix (which would need N*P*Q*C*R*S elements).
 */
conv2d_status_t conv2d_workspace_bytes(conv2d_desc_t desc, size_t *bytes);

/*
 * Force a kernel family for later conv2d_forward_desc calls (tests and A/B
 * measurements).  CONV2D_ERR_UNSUPPORTED if the family cannot run this layer.
 */
conv2d_status_t conv2d_desc_set_algo(conv2d_desc_t desc, conv2d_algo_t algo);

/*
 * Describe the plan the chooser made for this layer (kernel family, tile and
 * grid) as a NUL-terminated string in buf (truncated to len bytes).
 */
conv2d_status_t conv2d_desc_plan(conv2d_desc_t desc, char *buf, size_t len);

/* Forward convolution for a descriptor's layer.  Tensors as described above. */
conv2d_status_t conv2d_forward_desc(conv2d_desc_t desc, const void *x, const void *w,
                                    const void *bias, void *y, cudaStream_t stream);

/*
 * One-shot forward convolution: the same as creating a descriptor for these
 * sizes and calling conv2d_forward_desc (plans are cached internally per
 * shape, dtype and layout).
 */
conv2d_status_t conv2d_forward(const void *x, const void *w, const void *bias, void *y,
                               int N, int C, int H, int W, int K, int R, int S,
                               int stride, int pad, int dil,
                               conv2d_dtype_t dtype, conv2d_layout_t layout,
                               cudaStream_t stream);

/*
 * MSCRED signature matrices, the input of the encoder's first convolution
 * ("GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
 * Extension", section "Why Signature Matrices Are Useful": pairwise
 * relationships of the signals over a time interval, at several interval
 * lengths; the definition is the one of the MSCRED paper the page cites):
 *
 *   out[b][c][i][j] = sum_{t = e-w}^{e-1} series[i][t] * series[j][t] / w,
 *   e = t_first + b, w = windows[c],
 *
 * for b < n_steps, c < n_windows, i, j < n_signals.  series: device fp32
 * [n_signals][T] row-major; out: device fp32 [n_steps][n_windows][n_signals]
 * [n_signals] (NCHW with C = n_windows), caller-owned, must not overlap
 * series; windows: HOST array of n_windows lengths (any order, repeats
 * allowed).  fp32 products accumulated with FMA, newest sample first, one
 * division by w.  Asynchronous on stream; allocates nothing.
 * CONV2D_ERR_INVALID_ARG unless 1 <= n_signals <= 128, T >= 1,
 * 1 <= n_windows <= 8, every window >= 1, max window <= t_first,
 * t_first + n_steps - 1 <= T, n_steps >= 1 and both pointers are device
 * memory of the current device; CONV2D_ERR_MISALIGNED for pointers that are
 * not 4-byte aligned; CONV2D_ERR_CUDA if the launch fails.
 */
conv2d_status_t conv2d_signature_matrices(const float *series, int n_signals, int T,
                                          const int *windows, int n_windows, int t_first,
                                          int n_steps, float *out, cudaStream_t stream);

/*
 * One ConvLSTM cell step with the gate non-linearities and the state update
 * fused into the gate convolution's epilogue (ConvLSTM as "GPU-Accelerating
 * MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch Extension" uses it,
 * section "Understanding MSCRED", the cell of the ConvLSTM paper its
 * References cite, without peephole terms):
 *
 *   z = conv2d(xh, w) + bias          stride 1, padding pad, dilation dil
 *   i, f, o = sigmoid(z[0:Ch]), sigmoid(z[Ch:2Ch]), sigmoid(z[2Ch:3Ch]); g = tanh(z[3Ch:4Ch])
 *   c_next = f * c_prev + i * g;      h_next = o * tanh(c_next)
 *
 * fp32, NCHW.  xh: [N][Cx+Ch][H][W], the step input x_t (channels 0..Cx-1)
 * followed by h_{t-1}; w: [4*Ch][Cx+Ch][R][S], gate-major (i, f, o, g);
 * bias: [4*Ch] or NULL; c_prev, c_next: [N][Ch][H][W]; h_next: image n starts
 * at h_next + n*h_img_stride and holds [Ch][H][W] (h_img_stride =
 * (Cx+Ch)*H*W with h_next = the h slice of the next step's xh buffer writes
 * h_t where the next step reads it).  The padding must keep H x W.  Runs on
 * the 3xTF32 tensor-core kernel (the gate convolution meets the fp32 bound);
 * the gates never reach memory.  All pointers device memory of the current
 * device, 4-byte aligned; outputs must not overlap the inputs.  Errors as
 * for conv2d_forward; CONV2D_ERR_UNSUPPORTED if no kernel variant fits.
 */
conv2d_status_t conv2d_convlstm_cell(const float *xh, const float *w, const float *bias,
                                     const float *c_prev, float *c_next, float *h_next,
                                     int N, int Cx, int Ch, int H, int W, int R, int S, int pad,
                                     int dil, long long h_img_stride, cudaStream_t stream);

/*
 * Output size of the transposed convolution: H = (P-1)*stride - 2*pad +
 * dil*(R-1) + 1 + out_pad, W likewise from Q and S.  out_pad in
 * [0, max(stride, dil)) picks among the sizes whose forward convolution gives
 * P x Q.  CONV2D_ERR_INVALID_ARG if anything is out of range or H, W < 1.
 */
conv2d_status_t conv2d_deconv_output_dims(int P, int Q, int R, int S, int stride, int pad, int dil,
                                          int out_pad, int *H, int *W);

/*
 * Transposed convolution forward ("deconvolution"), the MSCRED decoder's
 * up-sampling layer ("GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a
 * Custom PyTorch Extension", section "Understanding MSCRED": the decoder
 * reconstructs the signature matrices): the adjoint of conv2d_forward in its
 * input,
 *   y[n,c,h,w] = bias[c] + sum_{k,p,q,r,s : h = p*stride-pad+r*dil,
 *                w = q*stride-pad+s*dil} x[n,k,p,q] * w[k,c,r,s].
 * x: [N][K][P][Q]; w: [K][C][R][S] (the forward convolution's weights);
 * bias: [C] or NULL; y: [N][C][H][W] (conv2d_deconv_output_dims).  fp32 NCHW
 * (CONV2D_ERR_UNSUPPORTED for other dtypes / layouts), R, S <= 8.  A gather,
 * deterministic, no atomics, no workspace: layers with more than 8 output
 * channels run on the 3xTF32 tensor-core kernel, one launch per output
 * residue class (h mod stride, w mod stride); the others (and layers with a
 * residue class without taps) on FFMA kernels.  Results meet the fp32 bound
 * 1e-6 * (sum |x||w| + |bias|) either way.  Pointers: device memory of the
 * current device, 4-byte aligned; y must not overlap x, w or bias.
 * Asynchronous on stream.  Errors as for conv2d_forward.
 */
conv2d_status_t conv2d_deconv_forward(const void *x, const void *w, const void *bias, void *y,
                                      int N, int K, int P, int Q, int C, int R, int S, int stride,
                                      int pad, int dil, int out_pad, conv2d_dtype_t dtype,
                                      conv2d_layout_t layout, cudaStream_t stream);

/*
 * Process-wide overrides of the chooser, for tests and A/B measurements.
 * Each is -1 (not set: the chooser decides) or a value; they apply to every
 * later call in the process, on every thread.  At the first call that needs
 * them they are seeded from the environment variables named in brackets;
 * after that only conv2d_set_override changes them (the environment is not
 * read again, so the per-call path reads no environment).  A forced value
 * that does not fit a layer makes that layer's call return
 * CONV2D_ERR_UNSUPPORTED.
 */
typedef enum {
    CONV2D_OVR_DIRECT = 0,        /* [CONV2D_DIRECT] fp32 direct kernel: 1 force, 0 never */
    CONV2D_OVR_CC_TILE,           /* [CONV2D_CC_TILE] FFMA implicit-GEMM tile id */
    CONV2D_OVR_CC_SPLIT,          /* [CONV2D_CC_SPLIT] FFMA cluster split-K: 1, 2 or 4 */
    CONV2D_OVR_TC_BN,             /* [CONV2D_TC_BN] f16/bf16 tensor-core tile width: 64, 128, 256 */
    CONV2D_OVR_TC_KSUB,           /* [CONV2D_TC_KSUB] 64-channel k-blocks per pipeline stage */
    CONV2D_OVR_TC_IM2COL,         /* [CONV2D_TC_IM2COL] 1: 1x1 layers read x through the im2col map */
    CONV2D_OVR_TC_WINDOW,         /* [CONV2D_TC_WINDOW] 1: window (im2win) mode only, 0: never */
    CONV2D_OVR_TC_WINVAR,         /* [CONV2D_TC_WINVAR] window-mode variant id */
    CONV2D_OVR_TC_ROTATE,         /* [CONV2D_TC_ROTATE] 0: every CTA starts its k-loop at stage 0 */
    CONV2D_OVR_TF_VAR,            /* [CONV2D_TF_VAR] 3xTF32 variant id */
    CONV2D_OVR_FP32_TC,           /* [CONV2D_FP32_TC] 0: AUTO never runs fp32 on tensor cores */
    CONV2D_OVR_DECONV_TC,         /* [CONV2D_DECONV_TC] transposed conv: 1 tensor cores, 0 FFMA */
    CONV2D_OVR_GRID_CAP,          /* [CONV2D_GRID_CAP] persistent kernels launch at most this many
                                     CTAs (so small layers run several tiles per CTA) */
    CONV2D_OVR_TEST_WITHHOLD,     /* [CONV2D_TEST_WITHHOLD] test hook, 1: in the f16/bf16 im2col /
                                     plain tensor-core kernel, CTA 0 never issues the loads of its
                                     first pipeline stage, so a bounded wait runs out: that CTA (and,
                                     in the 2-CTA kernel, its partner) writes none of its tiles, the
                                     call's device status becomes
                                     CONV2D_ERR_TIMEOUT, the kernel still returns and the context
                                     stays usable */
    CONV2D_OVR_TEST_WAIT_KCYCLES, /* [CONV2D_TEST_WAIT_KCYCLES] f16/bf16 tensor-core kernels: a bounded
                                     wait gives up after this many thousand SM cycles (default
                                     4,000,000, about 2 s) */
    CONV2D_OVR_TC_CTA2,           /* [CONV2D_TC_CTA2] f16/bf16 im2col / plain kernel: 1 only its 2-CTA
                                     variants (clusters of two CTAs issuing 2-CTA MMAs, M = 256, each
                                     CTA loading half of the weight tile), 0 never; unset, the
                                     chooser weighs them against the single-CTA variants */
    CONV2D_OVR_COUNT
} conv2d_override_t;

/* Set an override (value -1 clears it).  CONV2D_ERR_INVALID_ARG for an
 * unknown key or a value below -1.  Plans made before the change are
 * discarded. */
conv2d_status_t conv2d_set_override(conv2d_override_t key, int value);

/* Current value of an override (-1 if not set). */
conv2d_status_t conv2d_get_override(conv2d_override_t key, int *value);

/* Kernel families with compiled variants (tile shapes, pipeline depths). */
typedef enum {
    CONV2D_FAMILY_CUDA_CORE_TILE = 0,   /* FFMA implicit-GEMM tiles (CONV2D_OVR_CC_TILE ids) */
    CONV2D_FAMILY_TENSOR_CORE = 1,      /* f16/bf16 im2col / plain kernel: (BN, KSUB) pairs */
    CONV2D_FAMILY_TENSOR_CORE_WINDOW = 2, /* f16/bf16 window kernel (CONV2D_OVR_TC_WINVAR ids) */
    CONV2D_FAMILY_TF32X3 = 3,           /* fp32 3xTF32 kernel (CONV2D_OVR_TF_VAR ids) */
    CONV2D_FAMILY_TENSOR_CORE_PAIR = 4  /* f16/bf16 2-CTA im2col / plain kernel: (BN, KSUB) pairs */
} conv2d_family_t;

/* Number of compiled variants of a family (tests cover every one). */
conv2d_status_t conv2d_variant_count(conv2d_family_t family, int *count);

/*
 * Throughput probes (measurement only, not part of the convolution path):
 * one launch on `stream` of a kernel that does nothing but
 *   CONV2D_PEAK_FFMA      fp32 FMAs in registers (8 CTAs of 256 threads per SM),
 *   CONV2D_PEAK_TF32_MMA  tcgen05.mma kind::tf32, M=128 N=256 K=8, one CTA per SM,
 *   CONV2D_PEAK_BF16_MMA  tcgen05.mma kind::f16 (bf16), M=128 N=256 K=16,
 * `iters` rounds of them (1 .. 2^24), operands on chip.  *flops receives the
 * floating-point operations the launch performs (2 per multiply-add); the
 * caller times the launch with CUDA events.  CONV2D_ERR_UNSUPPORTED for the
 * MMA probes on a GPU other than sm_103; CONV2D_ERR_CUDA if the launch fails.
 */
typedef enum {
    CONV2D_PEAK_FFMA = 0,
    CONV2D_PEAK_TF32_MMA = 1,
    CONV2D_PEAK_BF16_MMA = 2
} conv2d_peak_kind_t;

conv2d_status_t conv2d_peak_probe(conv2d_peak_kind_t kind, int iters, cudaStream_t stream,
                                  double *flops);

/* Static text for a status code. */
const char *conv2d_status_string(conv2d_status_t status);

/*
 * Synchronise the current device, then read and clear the device status word
 * that kernels set when a bounded wait runs out.  CONV2D_OK if nothing was
 * recorded; CONV2D_ERR_TIMEOUT otherwise; CONV2D_ERR_CUDA if the
 * synchronisation itself failed.
 */
conv2d_status_t conv2d_get_device_status(void);

/* Library version, major*10000 + minor*100 + patch. */
int conv2d_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CONV2D_GB300_H */
