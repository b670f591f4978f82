// CUDA-core (FFMA) implicit-GEMM convolution: every dtype and layout.
//
// This is the full-precision CUDA-core path of "Enabling Memory-efficient
// Im2win Convolution with Multi-precision Support on GPU CUDA and Tensor
// Cores" (abstract) and the shared-memory kernel of "GPU-Accelerating MSCRED
// with CUDA, im2col, GEMM, and a Custom PyTorch Extension" (section "Global
// Memory and Shared Memory": stage reusable tiles in shared memory and reuse
// them across the threads of a block).  The GEMM view is the page's
// "Output matrix = Weight matrix x im2col(Input)" (section "Transforming
// Conv2D into im2col and GEMM"), but the im2col matrix is never built: each
// CTA gathers the BM x BK slice of it that it needs straight from x into
// shared memory, with zero fill for padding taps.
//
// GEMM view:  D[m, k] = sum_j A[m, j] * B[k, j]
//   m = (n, p, q) flattened output pixel, k = output channel,
//   j = reduction index; NCHW orders j as (c, r, s) (matching KCRS weights),
//   NHWC as (r, s, c) (matching KRSC weights), so B rows are contiguous.
//
// Per CTA: a BM x BN output tile; per thread: TM x TN accumulators in fp32.
// A per-layer table in shared memory maps each j to (element offset of the
// tap relative to the window origin, r*dil, s*dil), so a gathered element
// costs one table read, two bounds compares and one predicated load.
// Operands are widened to fp32 on the way into shared memory; the epilogue
// adds the bias, rounds once to the output type and stores through shared
// memory so that global writes are coalesced.
//
// Split-K (SPLIT = 2 or 4, fp32): layers with few output tiles but a long
// reduction launch SPLIT CTAs per tile as one thread-block cluster; each CTA
// reduces a contiguous slice of the k-tiles, parks its partial tile in its
// shared memory, and after a cluster barrier each CTA sums one slice of rows
// across the cluster through distributed shared memory and writes it.  No
// global workspace, and the summation order is fixed (deterministic).

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstdio>
#include <type_traits>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

struct CcParams {
    const void *x, *w, *bias;
    void *y;
    int N, C, H, W, K, R, S, stride, pad, dil, P, Q;
    int Kg;        // C*R*S (fits int: checked on the host)
    int64_t M;     // N*P*Q
};

// Table entry for reduction index j: offset of x[.., c, h0+dh, w0+dw] from
// x[.., 0, h0, w0] within one image, and the tap's (dh, dw).
struct Tap {
    int delta;
    short dh, dw;
};

// Taps held in shared memory at once (32 KB); a multiple of every BK.
constexpr int kTableChunk = 4096;

template <typename T, int LAYOUT, int BM, int BN, int BK, int TM, int TN>
struct CcCfg {
    static constexpr int NT = (BM / TM) * (BN / TN);
    static constexpr int TPB = NT / BM;               // threads per output row m
    static constexpr int A_PER = BK / TPB;            // A elements per thread per tile
    static constexpr int B_PER = (BN * BK) / NT;      // B elements per thread per tile
    static constexpr int AS = BM + 4;                 // padded row lengths (floats)
    static constexpr int BS = BN + 4;
    static constexpr int TMV = TM / 4, TNV = TN / 4;  // float4 groups per thread
    static_assert(NT % BM == 0, "one output row per thread for the gather");
    static_assert(BK % TPB == 0, "");
    static_assert((BN * BK) % NT == 0, "");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "");
    static constexpr size_t tile_floats = 2 * (size_t)BK * AS + 2 * (size_t)BK * BS;
    static constexpr size_t epi_floats =
        LAYOUT == CONV2D_NCHW ? (size_t)BN * (BM + 1) : (size_t)BM * (BN + 1);
    static constexpr size_t main_floats = tile_floats > epi_floats ? tile_floats : epi_floats;
};

template <typename T, int LAYOUT, int BM, int BN, int BK, int TM, int TN, int SPLIT>
__global__ void __launch_bounds__(CcCfg<T, LAYOUT, BM, BN, BK, TM, TN>::NT)
cc_conv_kernel(const CcParams p) {
    using Cfg = CcCfg<T, LAYOUT, BM, BN, BK, TM, TN>;
    constexpr int NT = Cfg::NT, TPB = Cfg::TPB, A_PER = Cfg::A_PER, B_PER = Cfg::B_PER;
    constexpr int AS = Cfg::AS, BS = Cfg::BS, TMV = Cfg::TMV, TNV = Cfg::TNV;

    extern __shared__ __align__(16) float smem[];
    float *As = smem;                          // [2][BK][AS]
    float *Bs = smem + 2 * BK * AS;            // [2][BK][BS]
    Tap *taps = reinterpret_cast<Tap *>(smem + Cfg::main_floats);   // [Kg]

    const T *__restrict__ x = static_cast<const T *>(p.x);
    const T *__restrict__ w = static_cast<const T *>(p.w);
    const int tid = threadIdx.x;
    // no early trigger: a kernel of many short CTAs lets the next one launch
    // at its exit, so the next grid is spread over idle SMs
    sm103a::pdl_wait();                        // the previous kernel's writes are visible
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;
    const int Kg = p.Kg;
    const int PQ = p.P * p.Q;
    // k-tiles this CTA reduces (all of them unless split across a cluster)
    const int KT_all = (Kg + BK - 1) / BK;
    int split_rank = 0;
    if (SPLIT > 1) split_rank = (int)cooperative_groups::this_cluster().block_rank();
    const int kt_begin = (int)((int64_t)KT_all * split_rank / SPLIT);
    const int kt_end = (int)((int64_t)KT_all * (split_rank + 1) / SPLIT);

    // Reduction-index table, built for kTableChunk indices at a time.
    auto build_taps = [&](int jbase) {
        const int jend = min(Kg, jbase + kTableChunk);
        for (int j = jbase + tid; j < jend; j += NT) {
            int c, r, s;
            if (LAYOUT == CONV2D_NCHW) {
                c = j / (p.R * p.S);
                int rs = j - c * p.R * p.S;
                r = rs / p.S;
                s = rs - r * p.S;
            } else {
                r = j / (p.S * p.C);
                int sc = j - r * p.S * p.C;
                s = sc / p.C;
                c = sc - s * p.C;
            }
            Tap t;
            t.dh = (short)(r * p.dil);
            t.dw = (short)(s * p.dil);
            t.delta = LAYOUT == CONV2D_NCHW ? (c * p.H + t.dh) * p.W + t.dw
                                            : (t.dh * p.W + t.dw) * p.C + c;
            taps[j - jbase] = t;
        }
    };
    build_taps((kt_begin * BK / kTableChunk) * kTableChunk);

    // This thread gathers A rows for output pixel m_ld.
    const int ml = tid % BM;
    const int kl0 = tid / BM;
    const int64_t m_ld = m0 + ml;
    const bool m_ok = m_ld < p.M;
    int ih0 = 0, iw0 = 0;
    int64_t xbase = 0;       // element offset of the window origin (may be "negative")
    int64_t ybase = 0;       // NCHW: offset of y[n, 0, p, q]
    if (m_ok) {
        int n = (int)(m_ld / PQ);
        int pq = (int)(m_ld - (int64_t)n * PQ);
        int pp = pq / p.Q, qq = pq - pp * p.Q;
        ih0 = pp * p.stride - p.pad;
        iw0 = qq * p.stride - p.pad;
        if (LAYOUT == CONV2D_NCHW) {
            xbase = (int64_t)n * p.C * p.H * p.W + (int64_t)ih0 * p.W + iw0;
            ybase = (int64_t)n * p.K * PQ + pq;
        } else {
            xbase = ((int64_t)n * p.H * p.W + (int64_t)ih0 * p.W + iw0) * p.C;
        }
    }
    __syncthreads();

    float a_reg[A_PER];
    float b_reg[B_PER];

    auto load_tile = [&](int kt) {
        const int j0 = kt * BK;
#pragma unroll
        for (int i = 0; i < A_PER; ++i) {
            const int j = j0 + kl0 + i * TPB;
            float v = 0.f;
            if (m_ok && j < Kg) {
                const Tap t = taps[j % kTableChunk];
                const int h = ih0 + t.dh, ww = iw0 + t.dw;
                if ((unsigned)h < (unsigned)p.H && (unsigned)ww < (unsigned)p.W)
                    v = to_f32<T>(__ldg(x + (xbase + t.delta)));
            }
            a_reg[i] = v;
        }
#pragma unroll
        for (int i = 0; i < B_PER; ++i) {
            const int e = tid + i * NT;
            const int kl = e % BK, nl = e / BK;
            const int j = j0 + kl, k = n0 + nl;
            float v = 0.f;
            if (j < Kg && k < p.K) v = to_f32<T>(__ldg(w + ((int64_t)k * Kg + j)));
            b_reg[i] = v;
        }
    };
    auto store_tile = [&](int buf) {
        float *as = As + buf * BK * AS;
        float *bs = Bs + buf * BK * BS;
#pragma unroll
        for (int i = 0; i < A_PER; ++i) as[(kl0 + i * TPB) * AS + ml] = a_reg[i];
#pragma unroll
        for (int i = 0; i < B_PER; ++i) {
            const int e = tid + i * NT;
            bs[(e % BK) * BS + e / BK] = b_reg[i];
        }
    };

    // column pairs (2jj, 2jj + 1) of row i, packed for fma.rn.f32x2 (two fp32
    // FMAs, each rounded as fmaf, in one issue slot)
    static_assert(TN % 2 == 0, "packed accumulator pairs");
    uint64_t acc2[TM][TN / 2];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int jj = 0; jj < TN / 2; ++jj) acc2[i][jj] = 0ull;

    const int tx = tid % (BN / TN);
    const int ty = tid / (BN / TN);
    if (kt_begin < kt_end) {
        load_tile(kt_begin);
        store_tile(0);
    }
    __syncthreads();
    for (int kt = kt_begin; kt < kt_end; ++kt) {
        const int cur = (kt - kt_begin) & 1;
        if (kt + 1 < kt_end) {
            if (((kt + 1) * BK) % kTableChunk == 0) {   // next tile starts a new table chunk
                __syncthreads();
                build_taps((kt + 1) * BK);
                __syncthreads();
            }
            load_tile(kt + 1);
        }
        const float *as = As + cur * BK * AS;
        const float *bs = Bs + cur * BK * BS;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int v = 0; v < TMV; ++v) {
                const float4 t = *reinterpret_cast<const float4 *>(as + kk * AS + v * (BM / TMV) + ty * 4);
                a[4 * v] = t.x; a[4 * v + 1] = t.y; a[4 * v + 2] = t.z; a[4 * v + 3] = t.w;
            }
#pragma unroll
            for (int v = 0; v < TNV; ++v) {
                const float4 t = *reinterpret_cast<const float4 *>(bs + kk * BS + v * (BN / TNV) + tx * 4);
                b[4 * v] = t.x; b[4 * v + 1] = t.y; b[4 * v + 2] = t.z; b[4 * v + 3] = t.w;
            }
            uint64_t b2[TN / 2];
#pragma unroll
            for (int jj = 0; jj < TN / 2; ++jj) b2[jj] = sm103a::pack_f32x2(b[2 * jj], b[2 * jj + 1]);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const uint64_t a2 = sm103a::pack_f32x2(a[i], a[i]);
#pragma unroll
                for (int jj = 0; jj < TN / 2; ++jj) acc2[i][jj] = sm103a::ffma2(a2, b2[jj], acc2[i][jj]);
            }
        }
        if (kt + 1 < kt_end) store_tile(cur ^ 1);
        __syncthreads();
    }
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int jj = 0; jj < TN / 2; ++jj) sm103a::unpack_f32x2(acc2[i][jj], acc[i][2 * jj], acc[i][2 * jj + 1]);

    // Epilogue: stage the tile in shared memory, then write coalesced rows.
    // The tile's bias values go to shared memory first: a global load placed
    // after a global store through a possibly aliasing pointer waits for it,
    // so bias loads inside the store loops would each cost a full latency.
    // (The barrier before the stores below publishes s_bias.)
    __shared__ float s_bias[BN];
    {
        const T *bias_g = static_cast<const T *>(p.bias);
        for (int j = tid; j < BN; j += NT)
            s_bias[j] = (bias_g && n0 + j < p.K) ? to_f32<T>(bias_g[n0 + j]) : 0.f;
    }
    float *cs = smem;
    if constexpr (SPLIT > 1) {
        // Partial tile -> own shared memory as cs[nl][ml]; cluster barrier;
        // CTA `split_rank` sums rows [lo, hi) of every CTA's partial tile.
        constexpr int CS = BM + 1;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int mi = (i / 4) * (BM / TMV) + ty * 4 + (i % 4);
                const int nj = (j / 4) * (BN / TNV) + tx * 4 + (j % 4);
                cs[nj * CS + mi] = acc[i][j];
            }
        auto cluster = cooperative_groups::this_cluster();
        cluster.sync();
        const float *parts[SPLIT];
#pragma unroll
        for (int r = 0; r < SPLIT; ++r) parts[r] = cluster.map_shared_rank(cs, r);
        T *y = static_cast<T *>(p.y);
        constexpr int ROWS = BM / SPLIT;
        const int lo = split_rank * ROWS;
        for (int e = tid; e < ROWS * BN; e += NT) {
            const int mi = lo + e % ROWS, nl = e / ROWS;
            const int64_t m = m0 + mi;
            const int k = n0 + nl;
            if (m < p.M && k < p.K) {
                float v = 0.f;
#pragma unroll
                for (int r = 0; r < SPLIT; ++r) v += parts[r][nl * CS + mi];
                v += s_bias[nl];
                if (LAYOUT == CONV2D_NCHW) {
                    const int n = (int)(m / PQ);
                    const int pq = (int)(m - (int64_t)n * PQ);
                    y[((int64_t)n * p.K + k) * PQ + pq] = from_f32<T>(v);
                } else {
                    y[m * p.K + k] = from_f32<T>(v);
                }
            }
        }
        cluster.sync();   // peers may still be reading this CTA's partial tile
        return;
    }
    T *y = static_cast<T *>(p.y);
    if (LAYOUT == CONV2D_NCHW) {
        // cs[nl][ml]: m contiguous, as in y[n][k][p][q].
        constexpr int CS = BM + 1;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int mi = (i / 4) * (BM / TMV) + ty * 4 + (i % 4);
                const int nj = (j / 4) * (BN / TNV) + tx * 4 + (j % 4);
                cs[nj * CS + mi] = acc[i][j];
            }
        __syncthreads();
        if (m_ok) {
            for (int nl = kl0; nl < BN; nl += TPB) {
                const int k = n0 + nl;
                if (k >= p.K) break;
                const float v = cs[nl * CS + ml] + s_bias[nl];
                y[ybase + (int64_t)k * PQ] = from_f32<T>(v);
            }
        }
    } else {
        // cs[ml][nl]: k contiguous, as in y[n][p][q][k].
        constexpr int CS = BN + 1;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int mi = (i / 4) * (BM / TMV) + ty * 4 + (i % 4);
                const int nj = (j / 4) * (BN / TNV) + tx * 4 + (j % 4);
                cs[mi * CS + nj] = acc[i][j];
            }
        __syncthreads();
        for (int e = tid; e < BM * BN; e += NT) {
            const int mi = e / BN, nl = e % BN;
            const int64_t m = m0 + mi;
            const int k = n0 + nl;
            if (m < p.M && k < p.K) {
                const float v = cs[mi * CS + nl] + s_bias[nl];
                y[m * p.K + k] = from_f32<T>(v);
            }
        }
    }
}

// ---------------------------------------------------------------- tile table

struct TileEntry {
    int BM, BN, BK, TM, TN;
    bool all_dtypes;   // instantiated for fp16 / bf16 too (otherwise fp32 only)
};
// Kept in sync with the dispatch switch below.
constexpr TileEntry kTiles[] = {
    {128, 64, 8, 8, 8, true},     // 0: 128 threads, 64 acc/thread
    {128, 128, 8, 8, 8, false},   // 1: 256 threads
    {64, 64, 16, 4, 4, true},     // 2: 256 threads, 16 acc/thread
    {128, 32, 16, 8, 4, false},   // 3: 128 threads (narrow K, e.g. 32 output channels)
    {64, 32, 16, 4, 4, false},    // 4: 128 threads
    {32, 32, 16, 4, 4, true},     // 5: 64 threads (tiny layers)
    {128, 128, 16, 8, 8, false},  // 6: 256 threads, deeper k-tile
    {128, 64, 16, 8, 8, false},   // 7: 128 threads, deeper k-tile
};
constexpr int kNumTiles = sizeof(kTiles) / sizeof(kTiles[0]);

// Split-K factors compiled for fp32 (tile ids 1, 6, 7, 2, 0).
bool split_compiled(int id, int split) {
    if (split == 1) return true;
    return (split == 2 || split == 4) && (id == 0 || id == 1 || id == 2 || id == 6 || id == 7);
}

template <typename T, int LAYOUT, int BM, int BN, int BK, int TM, int TN, int SPLIT>
conv2d_status_t launch_one(const Shape &s, const Tensors &t, int grid_m, int grid_n,
                           size_t smem, cudaStream_t st) {
    using Cfg = CcCfg<T, LAYOUT, BM, BN, BK, TM, TN>;
    auto kern = cc_conv_kernel<T, LAYOUT, BM, BN, BK, TM, TN, SPLIT>;
    // Opt in to >48 KB dynamic shared memory: raise the kernel's limit when a
    // launch needs more than was set before (per device).
    if (smem > 48 * 1024) {
        static std::atomic<int> set_bytes[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
        std::atomic<int> &cur = set_bytes[dev & 63];
        if (cur.load(std::memory_order_acquire) < (int)smem) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
                return CONV2D_ERR_CUDA;
            int prev = cur.load();
            while (prev < (int)smem && !cur.compare_exchange_weak(prev, (int)smem)) {
            }
        }
    }
    CcParams p;
    p.x = t.x; p.w = t.w; p.bias = t.bias; p.y = t.y;
    p.N = s.N; p.C = s.C; p.H = s.H; p.W = s.W; p.K = s.K; p.R = s.R; p.S = s.S;
    p.stride = s.stride; p.pad = s.pad; p.dil = s.dil; p.P = s.P; p.Q = s.Q;
    p.Kg = (int)s.Kg; p.M = s.M;
    if (SPLIT == 1) {
        if (launch_pdl(kern, dim3(grid_m, grid_n), dim3(Cfg::NT), smem, st, p) != cudaSuccess) {
            cudaGetLastError();
            return CONV2D_ERR_CUDA;
        }
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid_m, grid_n, SPLIT);
        cfg.blockDim = dim3(Cfg::NT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = SPLIT;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return CONV2D_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

template <typename T, int LAYOUT, int SPLIT>
conv2d_status_t dispatch_tile_split(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    const CudaCoreTile &c = pl.cc;
    const int gm = (int)((s.M + c.BM - 1) / c.BM);
    const int gn = (s.K + c.BN - 1) / c.BN;
    constexpr bool f32 = std::is_same<T, float>::value;
    switch (c.id) {
        case 0: return launch_one<T, LAYOUT, 128, 64, 8, 8, 8, SPLIT>(s, t, gm, gn, pl.smem_bytes, st);
        case 2: return launch_one<T, LAYOUT, 64, 64, 16, 4, 4, SPLIT>(s, t, gm, gn, pl.smem_bytes, st);
        case 5:
            if constexpr (SPLIT == 1)
                return launch_one<T, LAYOUT, 32, 32, 16, 4, 4, 1>(s, t, gm, gn, pl.smem_bytes, st);
            break;
        default: break;
    }
    if constexpr (f32) {
        switch (c.id) {
            case 1: return launch_one<T, LAYOUT, 128, 128, 8, 8, 8, SPLIT>(s, t, gm, gn, pl.smem_bytes, st);
            case 6: return launch_one<T, LAYOUT, 128, 128, 16, 8, 8, SPLIT>(s, t, gm, gn, pl.smem_bytes, st);
            case 7: return launch_one<T, LAYOUT, 128, 64, 16, 8, 8, SPLIT>(s, t, gm, gn, pl.smem_bytes, st);
            case 3:
                if constexpr (SPLIT == 1)
                    return launch_one<T, LAYOUT, 128, 32, 16, 8, 4, 1>(s, t, gm, gn, pl.smem_bytes, st);
                break;
            case 4:
                if constexpr (SPLIT == 1)
                    return launch_one<T, LAYOUT, 64, 32, 16, 4, 4, 1>(s, t, gm, gn, pl.smem_bytes, st);
                break;
            default: break;
        }
    }
    return CONV2D_ERR_INTERNAL;
}

template <typename T, int LAYOUT>
conv2d_status_t dispatch_tile(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    if constexpr (std::is_same<T, float>::value) {
        if (pl.cc.split == 2) return dispatch_tile_split<T, LAYOUT, 2>(s, pl, t, st);
        if (pl.cc.split == 4) return dispatch_tile_split<T, LAYOUT, 4>(s, pl, t, st);
    }
    if (pl.cc.split != 1) return CONV2D_ERR_INTERNAL;
    return dispatch_tile_split<T, LAYOUT, 1>(s, pl, t, st);
}

template <int LAYOUT>
conv2d_status_t dispatch_dtype(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    switch (s.dtype) {
        case CONV2D_F32: return dispatch_tile<float, LAYOUT>(s, pl, t, st);
        case CONV2D_F16: return dispatch_tile<__half, LAYOUT>(s, pl, t, st);
        case CONV2D_BF16: return dispatch_tile<__nv_bfloat16, LAYOUT>(s, pl, t, st);
    }
    return CONV2D_ERR_UNSUPPORTED;
}

}  // namespace

int cc_num_tiles() { return kNumTiles; }

bool cc_tile_available(int id, conv2d_dtype_t dtype, int split) {
    if (id < 0 || id >= kNumTiles) return false;
    if (dtype != CONV2D_F32) return kTiles[id].all_dtypes && split == 1;
    return split_compiled(id, split);
}

CudaCoreTile cc_tile(int id) {
    const TileEntry &e = kTiles[id];
    CudaCoreTile t;
    t.id = id;
    t.BM = e.BM; t.BN = e.BN; t.BK = e.BK; t.TM = e.TM; t.TN = e.TN;
    t.threads = (e.BM / e.TM) * (e.BN / e.TN);
    t.split = 1;
    return t;
}

// Tap offsets must fit in 32 bits (they are relative to one image).
bool cc_shape_ok(const Shape &s) {
    if (s.Kg >= (int64_t)1 << 31) return false;
    if ((int64_t)s.C * s.H * s.W >= (int64_t)1 << 31) return false;
    if ((int64_t)s.dil * (s.R - 1) > 32767 || (int64_t)s.dil * (s.S - 1) > 32767) return false;
    if ((int64_t)s.P * s.Q >= (int64_t)1 << 31) return false;
    return true;
}

size_t cc_smem_bytes(const Shape &s, const CudaCoreTile &t) {
    const size_t tile = 2 * (size_t)t.BK * (t.BM + 4) + 2 * (size_t)t.BK * (t.BN + 4);
    const size_t epi = s.layout == CONV2D_NCHW ? (size_t)t.BN * (t.BM + 1) : (size_t)t.BM * (t.BN + 1);
    const size_t main = tile > epi ? tile : epi;
    const size_t taps = s.Kg < kTableChunk ? (size_t)s.Kg : (size_t)kTableChunk;
    return main * sizeof(float) + taps * sizeof(Tap);
}

conv2d_status_t cc_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st) {
    if (s.layout == CONV2D_NCHW) return dispatch_dtype<CONV2D_NCHW>(s, p, t, st);
    return dispatch_dtype<CONV2D_NHWC>(s, p, t, st);
}

}  // namespace conv2d
