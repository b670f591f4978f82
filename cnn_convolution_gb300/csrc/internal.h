// Internal declarations shared by the host API and the kernel files of
// libconv2d_gb300.  Not part of the public ABI (see include/conv2d.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "conv2d.h"

namespace conv2d {

// One layer, fully validated; all derived sizes precomputed in 64 bits.
struct Shape {
    int N, C, H, W, K, R, S, stride, pad, dil;
    int P, Q;
    conv2d_dtype_t dtype;
    conv2d_layout_t layout;
    int64_t M;    // N*P*Q output pixels (GEMM rows)
    int64_t Kg;   // C*R*S reduction length
    int elt;      // element size in bytes
    int64_t x_elems() const { return (int64_t)N * C * H * W; }
    int64_t w_elems() const { return (int64_t)K * C * R * S; }
    int64_t y_elems() const { return (int64_t)N * K * P * Q; }
    double flops() const { return 2.0 * (double)M * K * (double)Kg; }
};

// Tile configurations of the CUDA-core implicit GEMM (index into a fixed table).
struct CudaCoreTile {
    int id;          // index into the kernel table
    int BM, BN, BK, TM, TN;
    int threads;
    int split;       // CTAs (one cluster) sharing one output tile's reduction
};

// Tile configurations of the tensor-core kernel.
struct TcTile {
    int BN;          // output channels per tile (multiple of 16, <= 256)
    int stages;      // smem pipeline depth
    int ksub = 1;    // 64-channel k-blocks per pipeline stage
    bool tma_store;  // epilogue through shared memory + TMA store
    bool force_im2col = false;   // 1x1 layers: use the im2col map even though a plain one would do
    bool window = false;         // stride-1 layers: one padded input window per channel block
    int win_variant = -1;        // index into the window-mode variant table
    bool rotate = true;          // CTA-dependent start of the k-loop
    bool cta2 = false;           // clusters of two CTAs issuing 2-CTA (M = 256) MMAs
};

// Variants of the fp32 split-precision (3xTF32) tensor-core kernel.
struct TfTile {
    int BN;          // output channels per tile
    int stages;      // smem pipeline depth (32 reduction elements per stage)
    int nprod;       // producer (gather + split) warps
    int id;          // index into the variant table
    int stage_ns;    // measured time of one 32-element stage of one tile (GB300)
    bool resb;       // the split weights of the CTA's output-channel tile stay resident
    int ngrp;        // producer groups: stage f is filled by group f % ngrp
    bool at;         // the A operand (split input) lives in tensor memory
};

enum class Algo { CudaCore, TensorCore, Tf32x3, Direct };

struct Plan {
    Algo algo;
    CudaCoreTile cc;
    TcTile tc;
    TfTile tf;
    int grid;        // CTAs launched
    int sm_count;
    size_t smem_bytes;
};

struct Tensors {
    const void *x;
    const void *w;
    const void *bias;
    void *y;
};

// CUDA-core path (any dtype / layout).  Returns CONV2D_OK or an error code.
int cc_num_tiles();
CudaCoreTile cc_tile(int id);
bool cc_tile_available(int id, conv2d_dtype_t dtype, int split);
bool cc_shape_ok(const Shape &s);
size_t cc_smem_bytes(const Shape &s, const CudaCoreTile &t);
conv2d_status_t cc_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st);

// Tensor-core path (f16/bf16, NHWC).
bool tc_shape_ok(const Shape &s, const Tensors *t);
size_t tc_smem_bytes(const TcTile &t);
int tc_stages(int bn, int ksub);   // 0 if the (BN, KSUB) variant does not exist
int tc_num_variants();             // compiled (BN, KSUB) variants of the plain / im2col kernel
int tc_cta2_stages(int bn, int ksub);
int tc_cta2_num_variants();   // stages of the 2-CTA variant (BN, KSUB), 0 if none
bool tc_window_ok(const Shape &s);
size_t tc_window_smem_bytes(const TcTile &t);
struct TcWinVariant {
    int bn, ksub, stages, win_kb, nwin;
    bool resident;
    int res_kb;
};
int tc_window_variants();
TcWinVariant tc_window_variant(int id);
bool tc_window_variant_ok(const Shape &s, int id);
conv2d_status_t tc_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st);

// Direct fp32 kernel for short reductions (C*R*S <= 64), either layout.
bool dc_shape_ok(const Shape &s);
size_t dc_smem_bytes(const Shape &s);
int dc_grid(const Shape &s);
void dc_block(int *rows, int *cols, int *threads, int *kc);   // the direct kernel's CTA block
conv2d_status_t dc_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st);

// fp32 tensor-core path (3xTF32 split precision, NCHW or NHWC).
bool tf_shape_ok(const Shape &s);
int tf_num_variants();
TfTile tf_variant(int id);
size_t tf_smem_bytes(const Shape &s, const TfTile &t);
// ConvLSTM-cell epilogue arguments of the 3xTF32 kernel (fp32, NCHW).
struct TfLstm {
    const float *c_prev;
    float *c_next;
    float *h_next;
    int64_t h_img;      // elements between images of h_next
};
// One residue class of a transposed convolution on the 3xTF32 kernel: the
// outputs (a + st*i, b + st*j) of y [N][C][H][W] gather input pixels
// (i + e[rj], j + f[sl]) with filter taps (r[rj], s[sl]), rj < J, sl < L.
struct TfDeconv {
    int H, W, a, b, st, J, L, R, S;
    int e[8], f[8], r[8], s[8];
};
bool tf_lstm_variant(int id);
conv2d_status_t tf_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st,
                          const TfLstm *lstm = nullptr, const TfDeconv *dv = nullptr);

// Transposed convolution, fp32 NCHW (arguments validated by the caller).
size_t dv_smem_bytes(int H, int W, int P, int Q, int C, int R, int S, int stride, int dil);
conv2d_status_t dv_launch(const float *x, const float *w, const float *bias, float *y, int N, int K,
                          int P, int Q, int C, int R, int S, int H, int W, int stride, int pad,
                          int dil, cudaStream_t st);

// MSCRED signature matrices (arguments validated by the caller).
conv2d_status_t sig_launch(const float *series, int n, int T, const int *windows, int n_windows,
                           int t_first, int n_steps, float *out, cudaStream_t st);

// Reciprocal for sm103a::fdiv: floor(2^32 / d) + 1, or 0 for d <= 1.
inline uint32_t recip_u32(int d) {
    return d <= 1 ? 0u : (uint32_t)((((uint64_t)1) << 32) / (uint64_t)d + 1);
}

// Launch with programmatic dependent launch (the kernel calls pdl_wait()
// before touching global memory); falls back to nothing else -- an error
// from the launch is returned as is.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Current value of a process-wide override (-1 = not set; see conv2d_set_override).
int ovr(conv2d_override_t key);

// Device status word (bounded-wait failures).
conv2d_status_t status_read_and_clear();
unsigned int *status_word_ptr();   // device address, per current device

}  // namespace conv2d
