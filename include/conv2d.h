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
 *  - dtype applies to x, w, bias and y alike.  CONV2D_F32 computes in fp32 on
 *    CUDA cores (FFMA, never TF32).  CONV2D_F16 / CONV2D_BF16 multiply in the
 *    input type and accumulate in fp32; y is rounded once, to nearest even.
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
