// Tensor-core implicit-GEMM convolution for sm_103a (fp16 / bf16, NHWC).
//
// The half-precision tensor-core path of "Enabling Memory-efficient Im2win
// Convolution with Multi-precision Support on GPU CUDA and Tensor Cores"
// (abstract: hardware half-precision multiply-accumulate fed by asynchronous
// data movement, with no im2col matrix in memory), written for Blackwell:
//
//   * GEMM view as in "GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a
//     Custom PyTorch Extension" (section "Transforming Conv2D into im2col and
//     GEMM"): D[m, k] = sum_{r,s,c} A[m, (r,s,c)] * W[k, (r,s,c)], with
//     m = (n, p, q) an output pixel and A[m, (r,s,c)] = x[n, p*st-pad+r*dil,
//     q*st-pad+s*dil, c] (zero outside the image).
//   * A tiles (128 output pixels x 64 channels at one filter tap (r, s)) are
//     fetched by TMA in im2col mode straight from x: the tensor map walks the
//     output pixels of the tile across rows and images, applies the conv
//     stride, the tap offset (s*dil, r*dil) and zero fill for padding.  B tiles
//     (BN output channels x 64 channels of w[k][r][s][c]) come from a tiled
//     tensor map.  Both land in shared memory with the 128-byte swizzle the
//     MMA descriptors expect.  No workspace exists.
//   * One thread issues tcgen05.mma (kind::f16, M=128, N=BN, K=16) into a
//     fp32 accumulator in tensor memory; tcgen05.commit frees each shared
//     memory stage and signals a finished accumulator.
//   * Persistent CTAs (one per SM) loop over output tiles; up to four
//     accumulators in tensor memory let the main loop run ahead while the
//     epilogue of earlier tiles (tcgen05.ld, + bias, one round-to-nearest-even
//     cast, then TMA stores of each warp's 32-row boxes, or in window mode
//     16-byte stores of each pixel's outputs straight into y) drains.
//   * 2-CTA variants of the im2col / plain kernel run as clusters of two
//     CTAs issuing tcgen05.mma.cta_group::2 (M=256): each CTA loads its own
//     A tile and half of the weight tile.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = tensor-memory
// allocator and MMA issuer, warps 2..5 = epilogue (warp w reads accumulator
// lanes 32*(w%4) .. 32*(w%4)+31, the lane quarter that warp may access).
//
// Every mbarrier wait is bounded: after kWaitLimitCycles the waiting thread sets
// a CTA abort flag and the device status word, every role drains what it
// started, tensor memory is freed, and the kernel returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

using namespace sm103a;

constexpr int kBM = 128;            // output pixels per tile (MMA M)
constexpr int kBK = 64;             // channels per k-block (128 bytes of fp16/bf16)
constexpr int kThreads = 192;
constexpr int kATileBytes = kBM * kBK * 2;

// D(tmem) (+)= A(smem) * B(smem)^T, M=128, N from idesc, K=16 per MMA.
// One 64-channel k-block: four MMAs (K = 16 each) at descriptor low words
// a_lo, b_lo advanced by 32 bytes per step; the first accumulates only if
// `accumulate` is set, the other three always.  One asm statement, 32-bit
// descriptor arithmetic: the single issuing thread's loop is on the critical
// path when an MMA takes ~50 cycles (N = 64).
__device__ __forceinline__ void mma4_f16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3, b1, b2, b3;\n\t"
        ".reg .b64 da0, da1, da2, da3, db0, db1, db2, db3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %3, %3;\n\t"
        "add.u32 a1, %1, 2;\n\tadd.u32 a2, %1, 4;\n\tadd.u32 a3, %1, 6;\n\t"
        "add.u32 b1, %2, 2;\n\tadd.u32 b2, %2, 4;\n\tadd.u32 b3, %2, 6;\n\t"
        "mov.b64 da0, {%1, %5};\n\tmov.b64 da1, {a1, %5};\n\tmov.b64 da2, {a2, %5};\n\tmov.b64 da3, {a3, %5};\n\t"
        "mov.b64 db0, {%2, %5};\n\tmov.b64 db1, {b1, %5};\n\tmov.b64 db2, {b2, %5};\n\tmov.b64 db3, {b3, %5};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da0, db0, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da1, db1, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da2, db2, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da3, db3, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kDescHi)
        : "memory");
}

// The same k-block for the 2-CTA (M = 256) MMA.
__device__ __forceinline__ void mma4_f16_2cta(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3, b1, b2, b3;\n\t"
        ".reg .b64 da0, da1, da2, da3, db0, db1, db2, db3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %3, %3;\n\t"
        "add.u32 a1, %1, 2;\n\tadd.u32 a2, %1, 4;\n\tadd.u32 a3, %1, 6;\n\t"
        "add.u32 b1, %2, 2;\n\tadd.u32 b2, %2, 4;\n\tadd.u32 b3, %2, 6;\n\t"
        "mov.b64 da0, {%1, %5};\n\tmov.b64 da1, {a1, %5};\n\tmov.b64 da2, {a2, %5};\n\tmov.b64 da3, {a3, %5};\n\t"
        "mov.b64 db0, {%2, %5};\n\tmov.b64 db1, {b1, %5};\n\tmov.b64 db2, {b2, %5};\n\tmov.b64 db3, {b3, %5};\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da0, db0, %3, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da1, db1, %3, q;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da2, db2, %3, q;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da3, db3, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kDescHi)
        : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulate, A and B K-major.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int n, int m = kBM) {
    return (1u << 4)                                   // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                   // A format: f16 / bf16
           | ((bf16 ? 1u : 0u) << 10)                  // B format
           | ((uint32_t)(n >> 3) << 17)                // N / 8
           | ((uint32_t)(m >> 4) << 24);               // M / 16 (256: a 2-CTA MMA)
}

// Accumulators in tensor memory: as many BN-column buffers as fit in 512
// columns, at most 4, so the MMAs can run up to 3 tiles ahead of the epilogue.
template <int BN> constexpr int tc_num_acc() { return 512 / BN >= 4 ? 4 : 512 / BN; }
template <int BN> constexpr uint32_t tc_tmem_cols() {
    return (uint32_t)(tc_num_acc<BN>() * BN) <= 256 ? 256u : 512u;
}
// The bias is staged once per CTA as fp32 in shared memory when K <= kBiasMax
// (8 KB with its 32-entry tail); larger layers read it from global memory.
constexpr int kBiasMax = 2016;
constexpr int kBiasBytes = (kBiasMax + 32) * 4;

__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <typename T> __device__ __forceinline__ float load_bias(const T *b, int k);
template <> __device__ __forceinline__ float load_bias<__half>(const __half *b, int k) {
    return __half2float(b[k]);
}
template <> __device__ __forceinline__ float load_bias<__nv_bfloat16>(const __nv_bfloat16 *b, int k) {
    return __bfloat162float(b[k]);
}

// Optional timeline trace of CTA 0 (compile with -DCONV2D_TC_TRACE; off in
// the library build): SM-cycle timestamps of the pipeline events, read back
// with conv2d_tc_trace_dump().
#ifdef CONV2D_TC_TRACE
__device__ unsigned long long g_tc_trace[4][8192];
__device__ unsigned int g_tc_trace_n[4];
// One tracing thread per role keeps its event count in a register and only
// stores (no atomics, nothing the thread waits for).
#define TC_TRACE(role, tag)                                                                  \
    do {                                                                                     \
        if (blockIdx.x == 0) {                                                               \
            if (tr_n[role] < 8192u)                                                          \
                g_tc_trace[role][tr_n[role]] =                                               \
                    ((unsigned long long)(tag) << 48) | ((unsigned long long)clock64() & 0xFFFFFFFFFFFFull); \
            ++tr_n[role];                                                                    \
            g_tc_trace_n[role] = tr_n[role];                                                 \
        }                                                                                    \
    } while (0)
#define TC_TRACE_DECL unsigned tr_n[4] = {0u, 0u, 0u, 0u}
#else
#define TC_TRACE(role, tag) \
    do {                    \
    } while (0)
#define TC_TRACE_DECL \
    do {              \
    } while (0)
#endif

struct TcParams {
    const void *bias;
    void *y;
    unsigned int *status;
    int64_t M;            // N*P*Q
    int K;                // output channels
    int PQ, Q;
    int stride, pad, dil;
    int S;                // filter width
    int CB;               // channel blocks of 64
    int KB;               // k-blocks per tile = R*S*CB
    int n_outer, n_inner; // k-block loop: outer x inner (see the producer)
    int chunked;          // 1x1 plain layer with C % 64 == 0: inner = channel blocks
    int rotate;           // start each CTA's k-loop at a different stage
    int n_tiles_n;        // tiles along K
    int total_tiles;
    // window mode only
    int P;                // output rows
    int R;                // filter height
    int Wp;               // padded row length W + 2*pad (rows of the window)
    int TR;               // output rows per tile (TR * Wp <= 128)
    int tiles_per_img;    // ceil(P / TR)
    // bounded waits give up after this many SM cycles
    long long wait_limit;
    // test hook (plain kernel): CTA 0 never issues the loads of its first
    // stage, so its MMA warp's wait on that stage runs out
    int withhold;
    // 2-CTA kernel: work units of two vertically adjacent M tiles (same N tile)
    int pair_units;
};

// Shared-memory layout: STAGES stages, each holding KSUB k-blocks (the KSUB A
// tiles, then the KSUB B tiles, every tile 1024-byte aligned), the epilogue
// warps' store buffers, the fp32 bias, then the barriers.  A stage is the unit of producer /
// consumer hand-off.  Measured on GB300, TMA cost is per instruction and per
// stage rather than per byte, so a stage carries KSUB k-blocks and its B tiles
// (and, for 1x1 layers, its A tiles) arrive in ONE 3-D box each.
// CTA2: the 2-CTA kernel, whose CTAs each hold half of the weight tile's BN
// rows and one more barrier per accumulator (the partner's relay).
template <int BN, int KSUB, int STAGES, bool CTA2 = false>
struct TcSmem {
    static constexpr int kBTileBytes = (CTA2 ? BN / 2 : BN) * kBK * 2;
    static constexpr int kStageBytes = KSUB * (kATileBytes + kBTileBytes);
    static constexpr int kAcc = tc_num_acc<BN>();
    // epilogue staging: per epilogue warp two buffers of 32 rows x 32 outputs
    // (64 B), 64-byte swizzled, for its own TMA stores
    static constexpr int kEpiBufBytes = 32 * 32 * 2;
    static constexpr size_t kEpiOffset = (size_t)STAGES * kStageBytes;
    // the layer's bias as fp32
    static constexpr size_t kBiasOffset = kEpiOffset + 4 * 2 * kEpiBufBytes;
    static constexpr size_t kBarOffset = kBiasOffset + kBiasBytes;
    // full[S], empty[S], acc_full[A], acc_empty[A], drain[1] (CTA2: +
    // partner_acc_empty[A]); then tmem addr, abort flag
    static constexpr size_t kBarBytes = (2 * STAGES + 2 * kAcc + 1 + (CTA2 ? kAcc : 0)) * 8;
    static constexpr size_t kBytes = kBarOffset + kBarBytes + 16 + 1024;   // +1024 for alignment
};

// A_TILE: the layer is a 1x1 / stride 1 / no padding convolution, so the A
// operand is x itself viewed as the [N*H*W, C] matrix and is fetched with a
// plain 2-D tiled map instead of an im2col one.
//
// CTA2: the kernel runs as clusters of two CTAs on neighbouring SMs that
// compute vertically adjacent M tiles of the same output-channel tile with
// 2-CTA MMAs (M = 256).  Each CTA loads its own A tile and its half of the
// weight tile (BN / 2 rows), so each SM takes in and serves 25 % (BN = 128)
// to 33 % (BN = 256) fewer bytes per k-block.  The even CTA's MMA thread
// issues every MMA once both CTAs' stage is full: both CTAs' copies of a
// stage (.cta_group::2 loads) count their bytes on the even CTA's full
// barrier, which the even CTA arms with the pair's total; the odd CTA's MMA
// warp, otherwise idle, relays its accumulator-empty events to the even CTA
// (a remote mbarrier arrival per tile); the even CTA's commits arrive on both
// CTAs' stage-empty and accumulator-full barriers.  Both CTAs walk
// the same sequence of stages.  Cluster barriers after the set-up and before
// the teardown keep either CTA from touching the other's barriers or
// tensor memory while it is not running.
template <typename T, int BN, int KSUB, int STAGES, bool A_TILE, bool CTA2>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmY, const TcParams p) {
    using L = TcSmem<BN, KSUB, STAGES, CTA2>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdesc = make_idesc(kBf16, BN, CTA2 ? 256 : 128);
    constexpr int kAcc = L::kAcc;
    constexpr uint32_t kTmemCols = tc_tmem_cols<BN>();

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_base + (uint32_t)L::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + kAcc + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * kAcc);
    // CTA2 only: in the even CTA, the odd CTA's relayed accumulator-empty events
    auto pacce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 * kAcc + 1 + a); };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kBarOffset + L::kBarBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBarOffset + L::kBarBytes + 4);
    auto a_tile = [&](int s, int j) {
        return smem_base + (uint32_t)(s * L::kStageBytes + j * kATileBytes);
    };
    auto b_tile = [&](int s, int j) {
        return smem_base + (uint32_t)(s * L::kStageBytes + KSUB * kATileBytes + j * L::kBTileBytes);
    };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    TC_TRACE_DECL;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 128);
            if (CTA2) mbar_init(pacce_bar(a), 1);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmY);
    }
    if (warp == 1) {
        if (CTA2) {
            tmem_alloc2(smem_u32(tmem_holder), kTmemCols);
            tmem_relinquish2();
        } else {
            tmem_alloc(smem_u32(tmem_holder), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // the partner's barriers exist before any remote arrival or commit reaches them
    if (CTA2) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();
    pdl_wait();                                // the previous kernel's writes are visible

    // Work units: one tile each, or (CTA2) two M tiles of one N tile, CTA
    // rank r of the pair taking M tile 2 * (u / n_tiles_n) + r.
    const uint32_t rank = CTA2 ? cluster_ctarank() : 0u;
    const int unit0 = CTA2 ? (int)blockIdx.x / 2 : (int)blockIdx.x;
    const int ustep = CTA2 ? (int)gridDim.x / 2 : (int)gridDim.x;
    const int n_units = CTA2 ? p.pair_units : p.total_tiles;
    auto unit_tm = [&](int u) { return CTA2 ? 2 * (u / p.n_tiles_n) + (int)rank : u / p.n_tiles_n; };

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        // k-blocks run as n_outer x n_inner: channel blocks x filter taps, or
        // (1x1 layers with C % 64 == 0) 1 x channel blocks.  A stage holds up to
        // KSUB consecutive inner k-blocks; its B tiles are one 3-D box of the
        // weight map (64 channels x BN outputs x KSUB taps or channel blocks)
        // and, for 1x1 layers, its A tiles are one 3-D box too.  This single
        // thread's loop is on the critical path: no divisions per k-block.
        int stage = 0;
        uint32_t phase = 0;
        uint32_t n_issued = 0;       // stages filled so far
        bool ok = true;
        const int dil = p.dil;
        // test hook: CTA 0 leaves its first stage empty (nothing armed, none of
        // its own copies in flight; in a pair the odd CTA's copies still land
        // on that barrier, whose phase then never completes)
        const bool held0 = p.withhold != 0 && blockIdx.x == 0;
        for (int u = unit0; u < n_units && ok; u += ustep) {
            const int tm = unit_tm(u);
            const int tn = u % p.n_tiles_n;
            const int64_t m0 = (int64_t)tm * kBM;
            const int n_img = (int)(m0 / p.PQ);
            const int pq = (int)(m0 - (int64_t)n_img * p.PQ);
            const int p0 = pq / p.Q, q0 = pq - p0 * p.Q;
            const int h0 = p0 * p.stride - p.pad;
            const int w0 = q0 * p.stride - p.pad;
            // this CTA's rows of the weight tile (CTA2: its half)
            const int k0 = tn * BN + (int)rank * (BN / 2);
            // Stages of a tile run in a CTA-dependent rotation (the same in
            // both CTAs of a pair), so that CTAs running at the same time fetch
            // different weight tiles instead of all hammering the same L2 lines.
            const int per_o = (p.n_inner + KSUB - 1) / KSUB;
            const int n_st = p.n_outer * per_o;
            const int rot = p.rotate ? (int)((unsigned)unit0 % (unsigned)n_st) : 0;
            if (A_TILE) {
                // 1x1 layers read x once: warm L2 with the A rows of this CTA's
                // next tile while this one streams (its boxes then hit L2)
                const int uf = u + ustep;
                if (uf < n_units && (int64_t)unit_tm(uf) * kBM < p.M) {
                    const int mf = unit_tm(uf) * kBM;
                    if (p.chunked)
                        for (int i0 = 0; i0 < p.n_inner; i0 += KSUB) tma_prefetch_tile_3d(&tmA, 0, mf, i0);
                    else
                        for (int o = 0; o < p.n_outer; ++o) tma_prefetch_tile_2d(&tmA, o * kBK, mf);
                }
            }
            for (int j = 0; j < n_st; ++j) {
                int sidx = rot + j;
                if (sidx >= n_st) sidx -= n_st;
                const int o = sidx / per_o;
                const int i0 = (sidx - o * per_o) * KSUB;
                const int nsub = min(KSUB, p.n_inner - i0);
                const int cx = p.chunked ? 0 : o * kBK;     // channel offset of this outer block
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
                TC_TRACE(3, 8);
                // CTA2: both CTAs' copies signal the even CTA's full barrier,
                // which the even CTA arms with the pair's byte count
                const uint32_t fb = CTA2 ? mapa_shared(full_bar(stage), 0) : full_bar(stage);
                const int a_tiles = (A_TILE && p.chunked) ? KSUB : nsub;
                if (!(held0 && n_issued == 0)) {
                    const uint32_t bytes = (uint32_t)(a_tiles * kATileBytes + KSUB * L::kBTileBytes);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), CTA2 ? 2u * bytes : bytes);
                    if (A_TILE) {
                        if (p.chunked) {
                            if constexpr (CTA2)
                                tma_load_tile_3d_cg2(a_tile(stage, 0), &tmA, fb, 0, (int)m0, i0);
                            else
                                tma_load_tile_3d(a_tile(stage, 0), &tmA, fb, 0, (int)m0, i0);
                        } else {
                            if constexpr (CTA2)
                                tma_load_tile_2d_cg2(a_tile(stage, 0), &tmA, fb, cx, (int)m0);
                            else
                                tma_load_tile_2d(a_tile(stage, 0), &tmA, fb, cx, (int)m0);
                        }
                    } else {
                        int r = i0 / p.S, s = i0 - r * p.S;
                        for (int jj = 0; jj < nsub; ++jj) {
                            if constexpr (CTA2)
                                tma_load_im2col_4d_cg2(a_tile(stage, jj), &tmA, fb, cx, w0, h0, n_img,
                                                       (uint16_t)(s * dil), (uint16_t)(r * dil));
                            else
                                tma_load_im2col_4d(a_tile(stage, jj), &tmA, fb, cx, w0, h0, n_img,
                                                   (uint16_t)(s * dil), (uint16_t)(r * dil));
                            if (++s == p.S) { s = 0; ++r; }
                        }
                    }
                    if constexpr (CTA2)
                        tma_load_tile_3d_cg2(b_tile(stage, 0), &tmB, fb, cx, k0, i0);
                    else
                        tma_load_tile_3d(b_tile(stage, 0), &tmB, fb, cx, k0, i0);
                }
                ++n_issued;
                TC_TRACE(0, 1);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && CTA2 && rank == 1) {
            // This CTA's copies signal the even CTA's barriers: give the ones
            // in flight time to land before the CTA goes away.
            const long long t0 = clock64();
            while (cycles_left(t0, p.wait_limit < (1ll << 20) ? p.wait_limit : (1ll << 20))) {
            }
        } else if (!ok) {
            // Let the copies already in flight land before the CTA goes away
            // (one time budget for all stages together).  Stage fill i went to
            // stage i % STAGES with phase (i / STAGES) & 1.
            const long long t0 = clock64();
            for (uint32_t i = n_issued > (uint32_t)STAGES ? n_issued - STAGES : 0; i < n_issued; ++i) {
                if (held0 && i == 0) continue;   // never armed: nothing to land
                while (!mbar_try_wait(full_bar((int)(i % STAGES)), (i / STAGES) & 1u) && cycles_left(t0, p.wait_limit)) {
                }
            }
        }
    } else if (CTA2 && rank == 1 && warp == 1 && lane == 0) {
        // ---------------------------------------------------------- relay (odd CTA)
        // The even CTA issues the pair's MMAs; this CTA's MMA thread tells it,
        // from the second use of each accumulator on, when this CTA's
        // epilogue has freed it.  (Stage-full events need no relay: this
        // CTA's copies signal the even CTA's barriers.)
        const uint32_t leader = 0;
        int acc = 0, n_tiles_done = 0;
        uint32_t acc_phase = 0;
        for (int u = unit0; u < n_units; u += ustep, ++n_tiles_done) {
            if (n_tiles_done >= kAcc) {
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_limit)) break;
                mbar_arrive_remote(mapa_shared(pacce_bar(acc), leader));
            }
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        // (CTA2: the even CTA's, for both CTAs)
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true, any = false;
        const uint32_t partner = 1;
        const uint32_t a_lo0 = desc_lo(a_tile(0, 0));
        const uint32_t b_lo0 = desc_lo(b_tile(0, 0));
        constexpr uint32_t kStageDesc = (uint32_t)(L::kStageBytes >> 4);   // 16-byte units
        constexpr uint32_t kADesc = (uint32_t)(kATileBytes >> 4);
        constexpr uint32_t kBDesc = (uint32_t)(L::kBTileBytes >> 4);
        for (int u = unit0; u < n_units && ok; u += ustep) {
            if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_limit) ||
                (CTA2 && !mbar_wait_cl(pacce_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_limit))) {
                ok = false;
                break;
            }
            TC_TRACE(1, 4);
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            const int per_o = (p.n_inner + KSUB - 1) / KSUB;
            const int n_st = p.n_outer * per_o;
            const int rot = p.rotate ? (int)((unsigned)unit0 % (unsigned)n_st) : 0;
            for (int j = 0; j < n_st; ++j) {
                int sidx = rot + j;
                if (sidx >= n_st) sidx -= n_st;
                const int o = sidx / per_o;
                const int nsub = min(KSUB, p.n_inner - (sidx - o * per_o) * KSUB);
                if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.wait_limit)) {
                    ok = false;
                    break;
                }
                TC_TRACE(1, 2);
                tc_fence_after();
                for (int jj = 0; jj < nsub; ++jj) {
                    const uint32_t a_lo = a_lo0 + (uint32_t)stage * kStageDesc + (uint32_t)jj * kADesc;
                    const uint32_t b_lo = b_lo0 + (uint32_t)stage * kStageDesc + (uint32_t)jj * kBDesc;
                    // four K = 16 steps, 32 bytes apart inside the swizzled rows
                    if constexpr (CTA2)
                        mma4_f16_2cta(d_tmem, a_lo, b_lo, kIdesc, (j | jj) != 0 ? 1u : 0u);
                    else
                        mma4_f16(d_tmem, a_lo, b_lo, kIdesc, (j | jj) != 0 ? 1u : 0u);
                }
                any = true;
                if (CTA2) {
                    // the stage is free in both CTAs once these MMAs are done
                    mma_commit2(empty_bar(stage));
                    mma_commit2(mapa_shared(empty_bar(stage), partner));
                } else {
                    mma_commit(empty_bar(stage));
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (CTA2) {
                mma_commit2(accf_bar(acc));
                mma_commit2(mapa_shared(accf_bar(acc), partner));
            } else {
                mma_commit(accf_bar(acc));
            }
            TC_TRACE(1, 3);
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
        }
        if (any) {
            // Make sure every MMA has retired before tensor memory is released.
            if (CTA2)
                mma_commit2(drain_bar);
            else
                mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain_bar, 0) && cycles_left(t0, p.wait_limit)) {
            }
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        // Thread = one output pixel (accumulator lane).  Per 32-output chunk:
        // tcgen05.ld -> + bias (fp32, staged once per CTA) -> one RN cast ->
        // the row's 64 bytes into the warp's own 64-byte-swizzled staging
        // buffer -> one TMA store of the warp's 32 x 32 box (clipped at M and
        // K).  Each warp alternates two buffers and orders its stores by
        // itself: no barrier between the epilogue warps per chunk.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        float *bias_s = reinterpret_cast<float *>(smem + L::kBiasOffset);
        const T *bias_g = static_cast<const T *>(p.bias);
        const bool bias_in_smem = bias_g != nullptr && p.K <= kBiasMax;
        if (bias_in_smem)
            for (int k = (int)threadIdx.x - 64; k < p.K; k += 128) bias_s[k] = load_bias<T>(bias_g, k);
        epilogue_bar_sync();                      // the staged bias is visible to the four warps
        const uint32_t wbuf = smem_base + (uint32_t)L::kEpiOffset + (uint32_t)(quarter * 2 * L::kEpiBufBytes);
        const uint32_t row_off = (uint32_t)lane * 64u;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);
        uint32_t chunk = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = unit0; u < n_units; u += ustep) {
            // One lane per warp waits, the whole warp follows (tcgen05.ld needs
            // a converged warp); then the four warps decide together, so that
            // if one warp's wait gave up they all leave the loop.
            int ok = 1;
            if (lane == 0) ok = mbar_wait(accf_bar(acc), acc_phase, abort_flag, p.status, p.wait_limit) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!epilogue_bar_all(ok != 0)) break;
            if (row == 0) TC_TRACE(2, 5);
            tc_fence_after();
            const int tm = unit_tm(u);
            const int tn = u % p.n_tiles_n;
            const int m_warp = tm * kBM + quarter * 32;
            const bool rows_in = (int64_t)m_warp < p.M;   // CTA2: the odd CTA's tile may lie past M
            const int k0 = tn * BN;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32cols(t_row + (uint32_t)c0, v);
                const int kc = k0 + c0;
                if (kc >= p.K) continue;            // uniform across the epilogue warps
                uint32_t o[16];
                const float4 *b4 = reinterpret_cast<const float4 *>(bias_s + kc);   // 128-byte aligned
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
                    float a2 = __uint_as_float(v[j + 2]), a3 = __uint_as_float(v[j + 3]);
                    if (bias_in_smem) {
                        const float4 bv = b4[j / 4];
                        a0 += bv.x;
                        a1 += bv.y;
                        a2 += bv.z;
                        a3 += bv.w;
                    } else if (bias_g != nullptr && kc + j < p.K) {
                        a0 += load_bias<T>(bias_g, kc + j);
                        a1 += load_bias<T>(bias_g, kc + j + 1);
                        a2 += load_bias<T>(bias_g, kc + j + 2);
                        a3 += load_bias<T>(bias_g, kc + j + 3);
                    }
                    o[j / 2] = pack2<T>(a0, a1);
                    o[j / 2 + 1] = pack2<T>(a2, a3);
                }
                const uint32_t buf = wbuf + (chunk & 1u) * (uint32_t)L::kEpiBufBytes;
                if (lane == 0) bulk_wait_read_le1();     // this warp's store from this buffer has read it
                __syncwarp();
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    st_shared_v4(buf + row_off + ((((uint32_t)g) ^ swz) << 4), o[4 * g], o[4 * g + 1],
                                 o[4 * g + 2], o[4 * g + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && rows_in) {
                    tma_store_2d(&tmY, buf, kc, m_warp);
                    bulk_commit_group();
                }
                ++chunk;
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive(acce_bar(acc));
            if (row == 0) TC_TRACE(2, 6);
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    // CTA2: the even CTA's MMAs (which write this CTA's tensor memory) have
    // drained and no arrival targets either CTA any more
    if (CTA2) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (CTA2)
            tmem_dealloc2(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ window (im2win) mode
//
// Stride-1 layers.  An M tile is TR whole rows of the *padded* output grid
// (TR * Wp <= 128 pixels, Wp = W + 2*pad): pixel j of the tile is output
// (p0 + j / Wp, j % Wp); columns j % Wp >= Q are computed and dropped.  In the
// padded, row-major flattening of the input, every filter tap (r, s) of such
// a tile reads the SAME pixels shifted by r*dil*Wp + s*dil rows.  So for each
// 64-channel block the kernel loads one window of TR + (R-1)*dil padded input
// rows (a tiled TMA box starting at column -pad: its out-of-image part is
// zero-filled, which is the padding) and runs the MMAs of all R*S taps on it,
// moving only the A descriptor's start row.  This is the memory-efficient
// im2win scheme of "Enabling Memory-efficient Im2win Convolution with
// Multi-precision Support on GPU CUDA and Tensor Cores" (abstract: windows
// with contiguous access for all kernel sizes), done by the copy engine:
// a 3x3 layer loads each input window once per channel block instead of
// nine 128-pixel im2col tiles.
//
// Shared memory: NWIN window slots of WINKB KB, the weight region, the fp32
// bias, barriers.  The weight region is either STAGES
// stages of KSUB weight tiles streamed per (tap group, channel block), or --
// RES, for layers whose whole weight tensor fits (one output-channel tile) --
// every weight tile of the layer, loaded once per CTA and kept resident; the
// pipeline then moves windows only.
template <int BN, int KSUB, int STAGES, int WINKB, int NWIN, bool RES, int RESKB>
struct TcWinSmem {
    static constexpr int kWinBytes = WINKB * 1024;     // (max row shift + 128) rows of 128 B
    static constexpr int kWinRows = kWinBytes / 128;
    static constexpr int kBTileBytes = BN * kBK * 2;
    static constexpr int kStageBytes = KSUB * kBTileBytes;
    static constexpr int kResBytes = RESKB * 1024;
    static constexpr size_t kStageOffset = (size_t)NWIN * kWinBytes;
    static constexpr int kAcc = tc_num_acc<BN>();
    static constexpr size_t kBiasOffset =
        kStageOffset + (RES ? (size_t)kResBytes : (size_t)STAGES * kStageBytes);
    static constexpr size_t kBarOffset = kBiasOffset + kBiasBytes;
    // full[S], empty[S], win_full[NWIN], win_empty[NWIN], acc_full[A], acc_empty[A], drain, resident
    static constexpr size_t kBarBytes = (2 * STAGES + 2 * NWIN + 2 * kAcc + 2) * 8;
    static constexpr size_t kBytes = kBarOffset + kBarBytes + 16 + 1024;
};

template <typename T, int BN, int KSUB, int STAGES, int WINKB, int NWIN, bool RES, int RESKB>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_window_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const TcParams p) {
    using L = TcWinSmem<BN, KSUB, STAGES, WINKB, NWIN, RES, RESKB>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdesc = make_idesc(kBf16, BN);
    constexpr int kAcc = L::kAcc;
    constexpr uint32_t kTmemCols = tc_tmem_cols<BN>();

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_base + (uint32_t)L::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto wfull_bar = [&](int w) { return bar_base + 8u * (2 * STAGES + w); };
    auto wempty_bar = [&](int w) { return bar_base + 8u * (2 * STAGES + NWIN + w); };
    auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 * NWIN + a); };
    auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 * NWIN + kAcc + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * NWIN + 2 * kAcc);
    const uint32_t res_bar = bar_base + 8u * (2 * STAGES + 2 * NWIN + 2 * kAcc + 1);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kBarOffset + L::kBarBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBarOffset + L::kBarBytes + 4);
    auto win_slot = [&](int w) { return smem_base + (uint32_t)(w * L::kWinBytes); };
    auto b_tile = [&](int s, int j) {
        return smem_base + (uint32_t)(L::kStageOffset + s * L::kStageBytes + j * L::kBTileBytes);
    };
    // resident weight tile of (channel block cb, tap t)
    auto res_tile = [&](int cb, int t) {
        return smem_base + (uint32_t)(L::kStageOffset + (cb * p.R * p.S + t) * L::kBTileBytes);
    };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int RS = p.R * p.S;
    TC_TRACE_DECL;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int w = 0; w < NWIN; ++w) {
            mbar_init(wfull_bar(w), 1);
            mbar_init(wempty_bar(w), 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        mbar_init(res_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();
    pdl_wait();                                // the previous kernel's writes are visible
    const uint32_t win_tx = (uint32_t)((p.TR + (p.R - 1) * p.dil) * p.Wp * 128);

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        int stage = 0, wslot = 0;
        uint32_t phase = 0, wphase = 0;
        uint32_t n_b = 0, n_w = 0;
        bool ok = true;
        bool res_issued = false;
        if (RES) {
            // every weight tile of the layer, one box per channel block
            mbar_arrive_expect_tx(res_bar, (uint32_t)(p.CB * RS * L::kBTileBytes));
            for (int cb = 0; cb < p.CB; ++cb)
                tma_load_tile_3d(res_tile(cb, 0), &tmB, res_bar, cb * kBK, 0, 0);
            res_issued = true;
        }
        for (int tile = blockIdx.x; tile < p.total_tiles && ok; tile += gridDim.x) {
            const int tm = tile / p.n_tiles_n;
            const int tn = tile - tm * p.n_tiles_n;
            const int n_img = tm / p.tiles_per_img;
            const int p0 = (tm - n_img * p.tiles_per_img) * p.TR;
            const int k0 = tn * BN;
            for (int cb = 0; cb < p.CB && ok; ++cb) {
                if (!mbar_wait(wempty_bar(wslot), wphase ^ 1u, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
                TC_TRACE(3, 8);
                mbar_arrive_expect_tx(wfull_bar(wslot), win_tx);
                tma_load_tile_4d(win_slot(wslot), &tmA, wfull_bar(wslot), cb * kBK, -p.pad, p0 - p.pad,
                                 n_img);
                TC_TRACE(0, 9);
                // Warm L2 with the window this CTA loads NWIN tiles later: its
                // smem load is issued only when a slot frees, and then reads
                // L2 instead of waiting on HBM.
                {
                    const int tf = tile + NWIN * (int)gridDim.x;
                    if (tf < p.total_tiles) {
                        const int tmf = tf / p.n_tiles_n;
                        const int nf = tmf / p.tiles_per_img;
                        const int pf = (tmf - nf * p.tiles_per_img) * p.TR;
                        tma_prefetch_tile_4d(&tmA, cb * kBK, -p.pad, pf - p.pad, nf);
                    }
                }
                ++n_w;
                if (++wslot == NWIN) { wslot = 0; wphase ^= 1u; }
                if (RES) continue;
                for (int t0 = 0; t0 < RS; t0 += KSUB) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, (uint32_t)(KSUB * L::kBTileBytes));
                    // one box: 64 channels x BN outputs x KSUB taps (taps past R*S read as zero)
                    tma_load_tile_3d(b_tile(stage, 0), &tmB, fb, cb * kBK, k0, t0);
                    TC_TRACE(0, 1);
                    ++n_b;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
        if (!ok) {
            // Let the copies already in flight land before the CTA goes away.
            const long long t0 = clock64();
            for (uint32_t i = n_b > (uint32_t)STAGES ? n_b - STAGES : 0; i < n_b; ++i)
                while (!mbar_try_wait(full_bar((int)(i % STAGES)), (i / STAGES) & 1u) && cycles_left(t0, p.wait_limit)) {
                }
            for (uint32_t i = n_w > (uint32_t)NWIN ? n_w - NWIN : 0; i < n_w; ++i)
                while (!mbar_try_wait(wfull_bar((int)(i % NWIN)), (i / NWIN) & 1u) && cycles_left(t0, p.wait_limit)) {
                }
            if (res_issued)
                while (!mbar_try_wait(res_bar, 0) && cycles_left(t0, p.wait_limit)) {
                }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        int stage = 0, wslot = 0, acc = 0;
        uint32_t phase = 0, wphase = 0, acc_phase = 0;
        bool ok = true, any = false;
        constexpr uint32_t kSubDesc32 = (uint32_t)(L::kBTileBytes >> 4);
        // window row shifts in descriptor units (16 bytes; a row is 128 bytes)
        const uint32_t a_col_step = (uint32_t)(p.dil * 8);
        const uint32_t a_row_step = (uint32_t)(p.dil * p.Wp * 8 - p.S * p.dil * 8);
        // 3x3 filters with resident weights: the nine taps' row shifts, once
        // per CTA, for a fully unrolled issue of each window's 36 MMAs
        const bool taps9 = RES && p.R == 3 && p.S == 3;
        uint32_t tap_off[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) tap_off[t] = (uint32_t)(((t / 3) * p.Wp + (t % 3)) * p.dil * 8);
        if (RES && !mbar_wait(res_bar, 0, abort_flag, p.status, p.wait_limit)) ok = false;
        for (int tile = blockIdx.x; tile < p.total_tiles && ok; tile += gridDim.x) {
            if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
            TC_TRACE(1, 4);
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int cb = 0; cb < p.CB && ok; ++cb) {
                if (!mbar_wait(wfull_bar(wslot), wphase, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
                TC_TRACE(1, 7);
                tc_fence_after();
                // Descriptors advance incrementally: tap (r, s) reads the
                // window's rows shifted by r*dil*Wp + s*dil pixels (8 descriptor
                // units of 16 bytes per 128-byte row), and the resident weight
                // tiles of consecutive taps are consecutive.  The start row need
                // not be a multiple of 8: the 128-byte swizzle follows absolute
                // shared-memory address bits, so the base-offset field stays 0.
                // The issuing thread's loop is on the critical path for N = 64
                // tiles (an MMA every ~50 cycles), so it does no multiplications.
                const uint32_t a_lo_w = desc_lo(win_slot(wslot));
                uint32_t a_tap = 0;                              // row shift of the tap, descriptor units
                int s = 0;
                uint32_t b_lo_res = RES ? desc_lo(res_tile(cb, 0)) : 0u;
                if (taps9) {
#pragma unroll
                    for (int t = 0; t < 9; ++t)
                        mma4_f16(d_tmem, a_lo_w + tap_off[t], b_lo_res + (uint32_t)t * kSubDesc32, kIdesc,
                                 (cb | t) != 0 ? 1u : 0u);
                    any = true;
                }
                for (int t0 = 0; t0 < RS && !taps9; t0 += KSUB) {
                    const int nsub = min(KSUB, RS - t0);
                    if (!RES) {
                        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.wait_limit)) { ok = false; break; }
                        TC_TRACE(1, 2);
                        tc_fence_after();
                    }
                    const uint32_t b_lo_stage = desc_lo(b_tile(stage, 0));
#pragma unroll 3
                    for (int j = 0; j < nsub; ++j) {
                        const uint32_t b_lo = RES ? b_lo_res : b_lo_stage + (uint32_t)j * kSubDesc32;
                        mma4_f16(d_tmem, a_lo_w + a_tap, b_lo, kIdesc, (cb | (t0 + j)) != 0 ? 1u : 0u);
                        if (RES) b_lo_res += kSubDesc32;
                        a_tap += a_col_step;
                        if (++s == p.S) { s = 0; a_tap += a_row_step; }
                    }
                    any = true;
                    if (!RES) {
                        mma_commit(empty_bar(stage));
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                }
                if (!ok) break;
                mma_commit(wempty_bar(wslot));
                if (++wslot == NWIN) { wslot = 0; wphase ^= 1u; }
            }
            if (!ok) break;
            mma_commit(accf_bar(acc));
            TC_TRACE(1, 3);
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
        }
        if (any) {
            mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain_bar, 0) && cycles_left(t0, p.wait_limit)) {
            }
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        // Accumulator lane j is padded-grid pixel (j / Wp, j % Wp) of the
        // tile's TR rows; lanes with j % Wp >= Q (or rows past P) are padding
        // columns and are dropped.  Each valid lane writes its pixel's outputs
        // straight into y, as in the im2col kernel.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int ti = row / p.Wp, tq = row - ti * p.Wp;
        const bool lane_valid = ti < p.TR && tq < p.Q;
        float *bias_s = reinterpret_cast<float *>(smem + L::kBiasOffset);
        const T *bias_g = static_cast<const T *>(p.bias);
        const bool bias_in_smem = bias_g != nullptr && p.K <= kBiasMax;
        if (bias_in_smem)
            for (int k = (int)threadIdx.x - 64; k < p.K; k += 128) bias_s[k] = load_bias<T>(bias_g, k);
        epilogue_bar_sync();                      // the staged bias is visible to the four warps
        T *y = static_cast<T *>(p.y);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
            int ok = 1;
            if (lane == 0) ok = mbar_wait(accf_bar(acc), acc_phase, abort_flag, p.status, p.wait_limit) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!epilogue_bar_all(ok != 0)) break;
            if (row == 0) TC_TRACE(2, 5);
            tc_fence_after();
            const int tm = tile / p.n_tiles_n;
            const int tn = tile - tm * p.n_tiles_n;
            const int n_img = tm / p.tiles_per_img;
            const int p0 = (tm - n_img * p.tiles_per_img) * p.TR;
            const int k0 = tn * BN;
            const bool valid = lane_valid && p0 + ti < p.P;
            const int64_t pix = ((int64_t)n_img * p.P + (valid ? p0 + ti : 0)) * p.Q + (valid ? tq : 0);
            T *yrow = y + pix * (int64_t)p.K;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32cols(t_row + (uint32_t)c0, v);
                const int kc = k0 + c0;
                if (kc >= p.K) continue;
                uint32_t o[16];
                const float4 *b4 = reinterpret_cast<const float4 *>(bias_s + kc);   // 128-byte aligned
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
                    float a2 = __uint_as_float(v[j + 2]), a3 = __uint_as_float(v[j + 3]);
                    if (bias_in_smem) {
                        const float4 bv = b4[j / 4];
                        a0 += bv.x;
                        a1 += bv.y;
                        a2 += bv.z;
                        a3 += bv.w;
                    } else if (bias_g != nullptr && kc + j < p.K) {
                        a0 += load_bias<T>(bias_g, kc + j);
                        a1 += load_bias<T>(bias_g, kc + j + 1);
                        a2 += load_bias<T>(bias_g, kc + j + 2);
                        a3 += load_bias<T>(bias_g, kc + j + 3);
                    }
                    o[j / 2] = pack2<T>(a0, a1);
                    o[j / 2 + 1] = pack2<T>(a2, a3);
                }
                if (valid) {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (kc + 8 * g < p.K)
                            st_global_v4(yrow + kc + 8 * g, o[4 * g], o[4 * g + 1], o[4 * g + 2], o[4 * g + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive(acce_bar(acc));
            if (row == 0) TC_TRACE(2, 6);
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using EncodeIm2colFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const int *, const int *,
                                    cuuint32_t, cuuint32_t, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

std::once_flag g_fn_once;
EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;

bool load_driver_fns() {
    std::call_once(g_fn_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<EncodeTiledFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(f);
    });
    return g_encode_tiled && g_encode_im2col;
}

struct TcMaps {
    alignas(64) CUtensorMap a, b, y;   // y: the im2col / plain kernel's store map
};

// Encode the tensor maps of a launch: x (im2col, plain matrix or window), w,
// and for the im2col / plain kernel y.
// Window geometry of a stride-1 layer (see the window kernel).
struct WinGeom {
    int Wp, TR, TRW, max_shift;
};
WinGeom win_geom(const Shape &s) {
    WinGeom g;
    g.Wp = s.W + 2 * s.pad;
    g.TR = g.Wp > 0 ? kBM / g.Wp : 0;
    g.TRW = g.TR + (s.R - 1) * s.dil;
    g.max_shift = (s.R - 1) * s.dil * g.Wp + (s.S - 1) * s.dil;
    return g;
}

// A 1x1 / stride 1 / no padding layer whose channel count is a multiple of 64:
// its k-blocks are channel blocks with a uniform 128-byte stride, so KSUB of
// them can be fetched as one box.
bool chunked_layer(const Shape &s, int amode) { return amode == 1 && s.C % kBK == 0; }

// amode: 0 = im2col A, 1 = plain [N*H*W, C] A, 2 = window A.
// B is a 3-D map: (64 channels, K outputs, KSUB taps) boxes over w viewed as
// (C, K, R*S) -- or, for chunked 1x1 layers, (64, K, C/64 channel blocks).
conv2d_status_t encode_maps(const Shape &s, int BN, int KSUB, int amode, const Tensors &t, TcMaps *m) {
    if (!load_driver_fns()) return CONV2D_ERR_CUDA;
    const CUtensorMapDataType dt =
        s.dtype == CONV2D_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool a_tile = amode == 1;
    if (amode == 2) {
        // x as (C, W, H, N); box = 64 channels x Wp columns x TRW rows x 1 image
        const WinGeom g = win_geom(s);
        const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
        const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2,
                                       (cuuint64_t)s.H * s.W * s.C * 2};
        const cuuint32_t box[4] = {kBK, (cuuint32_t)g.Wp, (cuuint32_t)g.TRW, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode_tiled(&m->a, dt, 4, const_cast<void *>(t.x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    } else if (a_tile && chunked_layer(s, amode)) {
        // x as (64 channels, N*H*W pixels, C/64 channel blocks)
        const cuuint64_t dims[3] = {(cuuint64_t)kBK, (cuuint64_t)s.N * s.H * s.W, (cuuint64_t)(s.C / kBK)};
        const cuuint64_t strides[2] = {(cuuint64_t)s.C * 2, (cuuint64_t)kBK * 2};
        const cuuint32_t box[3] = {kBK, kBM, (cuuint32_t)KSUB};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode_tiled(&m->a, dt, 3, const_cast<void *>(t.x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    } else if (a_tile) {
        const cuuint64_t dims[2] = {(cuuint64_t)s.C, (cuuint64_t)s.N * s.H * s.W};
        const cuuint64_t strides[1] = {(cuuint64_t)s.C * 2};
        const cuuint32_t box[2] = {kBK, kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (g_encode_tiled(&m->a, dt, 2, const_cast<void *>(t.x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    } else {
        const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
        const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2,
                                       (cuuint64_t)s.H * s.W * s.C * 2};
        // window origins span [-pad, extent - 1 + pad - dil*(ksize-1)] in W and H
        const int lower[2] = {-s.pad, -s.pad};
        const int upper[2] = {s.pad - s.dil * (s.S - 1), s.pad - s.dil * (s.R - 1)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)s.stride, (cuuint32_t)s.stride, 1};
        if (g_encode_im2col(&m->a, dt, 4, const_cast<void *>(t.x), dims, strides, lower, upper, kBK,
                            kBM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }
    if (chunked_layer(s, amode)) {
        // w as (64 channels, K outputs, C/64 channel blocks)
        const cuuint64_t dims[3] = {(cuuint64_t)kBK, (cuuint64_t)s.K, (cuuint64_t)(s.C / kBK)};
        const cuuint64_t strides[2] = {(cuuint64_t)s.C * 2, (cuuint64_t)kBK * 2};
        const cuuint32_t box[3] = {kBK, (cuuint32_t)BN, (cuuint32_t)KSUB};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode_tiled(&m->b, dt, 3, const_cast<void *>(t.w), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    } else {
        // w as (C channels, K outputs, R*S taps); w[k][r][s][c] = tap r*S+s
        const cuuint64_t dims[3] = {(cuuint64_t)s.C, (cuuint64_t)s.K, (cuuint64_t)s.R * s.S};
        const cuuint64_t strides[2] = {(cuuint64_t)s.R * s.S * s.C * 2, (cuuint64_t)s.C * 2};
        const cuuint32_t box[3] = {kBK, (cuuint32_t)BN, (cuuint32_t)KSUB};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode_tiled(&m->b, dt, 3, const_cast<void *>(t.w), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }
    if (amode != 2) {
        // y as the [M, K] row-major matrix; boxes of 32 rows x 32 outputs (one epilogue warp's store)
        const cuuint64_t dims[2] = {(cuuint64_t)s.K, (cuuint64_t)s.M};
        const cuuint64_t strides[1] = {(cuuint64_t)s.K * 2};
        const cuuint32_t box[2] = {32, 32};
        const cuuint32_t estr[2] = {1, 1};
        if (g_encode_tiled(&m->y, dt, 2, t.y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

// Maps depend only on the layer, the tile width, the A mode and the three
// pointers; repeated calls with the same tensors reuse them (host time).
struct MapKey {
    int v[15];
    const void *x, *w, *y;
    bool operator==(const MapKey &o) const {
        return std::memcmp(v, o.v, sizeof(v)) == 0 && x == o.x && w == o.w && y == o.y;
    }
};

conv2d_status_t cached_maps(const Shape &s, int BN, int KSUB, int amode, const Tensors &t,
                            const TcMaps **out) {
    constexpr int kSlots = 8;
    struct Slot {
        MapKey key;
        TcMaps maps;
        bool used = false;
    };
    thread_local Slot slots[kSlots];
    thread_local int next = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey k;
    const int vals[15] = {s.N, s.C, s.H, s.W, s.K, s.R, s.S, s.stride, s.pad, s.dil,
                          (int)s.dtype, BN, amode, dev, KSUB};
    std::memcpy(k.v, vals, sizeof(vals));
    k.x = t.x;
    k.w = t.w;
    k.y = t.y;
    for (int i = 0; i < kSlots; ++i) {
        if (slots[i].used && slots[i].key == k) {
            *out = &slots[i].maps;
            return CONV2D_OK;
        }
    }
    Slot &sl = slots[next];
    next = (next + 1) % kSlots;
    sl.used = false;
    conv2d_status_t st = encode_maps(s, BN, KSUB, amode, t, &sl.maps);
    if (st != CONV2D_OK) return st;
    sl.key = k;
    sl.used = true;
    *out = &sl.maps;
    return CONV2D_OK;
}

// cudaFuncSetAttribute once per device for one kernel; `done_mask` must be
// owned by that kernel (one static per template instantiation of the caller).
bool ensure_smem_attr(const void *kern, size_t bytes, std::atomic<uint64_t> &done_mask) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const uint64_t bit = (uint64_t)1 << (dev & 63);
    if (done_mask.load(std::memory_order_acquire) & bit) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return false;
    done_mask.fetch_or(bit, std::memory_order_release);
    return true;
}

// Bounded-wait limit and the stall test hook of a launch, from the overrides
// (the hook exists in the im2col / plain kernels, single-CTA and 2-CTA).
void set_wait_hooks(TcParams *p, bool has_withhold_hook) {
    const int kc = ovr(CONV2D_OVR_TEST_WAIT_KCYCLES);
    p->wait_limit = kc > 0 ? (long long)kc * 1000 : kWaitLimitCycles;
    p->withhold = has_withhold_hook && ovr(CONV2D_OVR_TEST_WITHHOLD) == 1 ? 1 : 0;
}

// Largest number of 2-CTA clusters of a kernel resident at once on this
// device (queried once per device and instantiation): a persistent 2-CTA
// launch must not exceed it, or the extra clusters would run after the others
// instead of beside them.
int max_pair_clusters(const void *kern, size_t smem, std::atomic<uint64_t> &done, std::atomic<int> *cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const uint64_t bit = (uint64_t)1 << dev;
    if (done.load(std::memory_order_acquire) & bit) return cache[dev].load(std::memory_order_relaxed);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    done.fetch_or(bit, std::memory_order_release);
    return n;
}

template <typename T, int BN, int KSUB, int STAGES, bool A_TILE, bool CTA2>
conv2d_status_t launch_tc(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    using L = TcSmem<BN, KSUB, STAGES, CTA2>;
    const TcMaps *maps = nullptr;
    // 2-CTA kernel: each CTA loads half of the weight tile, BN / 2 rows
    conv2d_status_t mst = cached_maps(s, CTA2 ? BN / 2 : BN, KSUB, A_TILE ? 1 : 0, t, &maps);
    if (mst != CONV2D_OK) return mst;
    TcParams p;
    p.bias = t.bias;
    p.y = t.y;
    p.status = status_word_ptr();
    set_wait_hooks(&p, true);
    p.M = s.M;
    p.K = s.K;
    p.PQ = s.P * s.Q;
    p.Q = s.Q;
    p.stride = s.stride;
    p.pad = s.pad;
    p.dil = s.dil;
    p.S = s.S;
    p.CB = (s.C + kBK - 1) / kBK;
    p.KB = s.R * s.S * p.CB;
    p.chunked = chunked_layer(s, A_TILE ? 1 : 0) ? 1 : 0;
    p.n_outer = p.chunked ? 1 : p.CB;
    p.n_inner = p.chunked ? p.CB : s.R * s.S;
    p.rotate = pl.tc.rotate ? 1 : 0;
    p.n_tiles_n = (s.K + BN - 1) / BN;
    const int64_t m_tiles = (s.M + kBM - 1) / kBM;
    const int64_t tiles = m_tiles * (int64_t)p.n_tiles_n;
    if (tiles > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    p.total_tiles = (int)tiles;
    p.pair_units = (int)(((m_tiles + 1) / 2) * p.n_tiles_n);
    auto kern = tc_conv_kernel<T, BN, KSUB, STAGES, A_TILE, CTA2>;
    static std::atomic<uint64_t> attr_done{0};   // this instantiation's per-device flags
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), L::kBytes, attr_done))
        return CONV2D_ERR_CUDA;
    int grid = pl.grid > 0 ? pl.grid : 1;
    if (!CTA2) {
        if (launch_pdl(kern, dim3(grid), dim3(kThreads), L::kBytes, st, maps->a, maps->b, maps->y, p) !=
            cudaSuccess) {
            cudaGetLastError();
            return CONV2D_ERR_CUDA;
        }
        return CONV2D_OK;
    }
    static std::atomic<uint64_t> occ_done{0};
    static std::atomic<int> occ[64];
    const int clusters = max_pair_clusters(reinterpret_cast<const void *>(kern), L::kBytes, occ_done, occ);
    if (clusters < 1) return CONV2D_ERR_UNSUPPORTED;
    grid = 2 * std::max(1, std::min(std::min(grid / 2, clusters), p.pair_units));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, maps->a, maps->b, maps->y, p) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

template <typename T, int BN, int KSUB, int STAGES, int WINKB, int NWIN, bool RES, int RESKB>
conv2d_status_t launch_tc_window(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    using L = TcWinSmem<BN, KSUB, STAGES, WINKB, NWIN, RES, RESKB>;
    const TcMaps *maps = nullptr;
    // resident weights arrive as one (64, BN, R*S) box per channel block
    conv2d_status_t mst = cached_maps(s, BN, RES ? s.R * s.S : KSUB, 2, t, &maps);
    if (mst != CONV2D_OK) return mst;
    const WinGeom g = win_geom(s);
    TcParams p;
    p.bias = t.bias;
    p.y = t.y;
    p.status = status_word_ptr();
    set_wait_hooks(&p, false);
    p.M = s.M;
    p.K = s.K;
    p.PQ = s.P * s.Q;
    p.Q = s.Q;
    p.stride = s.stride;
    p.pad = s.pad;
    p.dil = s.dil;
    p.S = s.S;
    p.CB = (s.C + kBK - 1) / kBK;
    p.KB = s.R * s.S * p.CB;
    p.n_tiles_n = (s.K + BN - 1) / BN;
    p.P = s.P;
    p.R = s.R;
    p.Wp = g.Wp;
    p.TR = g.TR;
    p.tiles_per_img = (s.P + g.TR - 1) / g.TR;
    const int64_t tiles = (int64_t)s.N * p.tiles_per_img * p.n_tiles_n;
    if (tiles > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    p.total_tiles = (int)tiles;
    auto kern = tc_conv_window_kernel<T, BN, KSUB, STAGES, WINKB, NWIN, RES, RESKB>;
    static std::atomic<uint64_t> attr_done{0};
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), L::kBytes, attr_done))
        return CONV2D_ERR_CUDA;
    const int grid = pl.grid > 0 ? pl.grid : 1;
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), L::kBytes, st, maps->a, maps->b, p) !=
        cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

// Variants: (BN, KSUB, STAGES) with about 192 KB of stages.
#define CONV2D_TC_VARIANTS(X) \
    X(64, 2, 4)               \
    X(64, 4, 2)               \
    X(128, 1, 6)              \
    X(128, 2, 3)              \
    X(128, 3, 2)              \
    X(256, 1, 4)              \
    X(256, 2, 2)

// 2-CTA variants of the im2col / plain kernel: (BN, KSUB, STAGES); a CTA's
// stage holds KSUB A tiles and KSUB half weight tiles (BN / 2 rows).
#define CONV2D_TC_CTA2_VARIANTS(X) \
    X(128, 2, 4)                   \
    X(128, 3, 2)                   \
    X(128, 4, 2)                   \
    X(256, 2, 3)

// Window-mode variants: (BN, KSUB, STAGES, window slot KB, window slots,
// resident weights, resident KB).  Id = position in this list.  The last two
// size their window slots to 3x3 and 5x5 layers of rows up to 32 pixels so
// that a third weight stage fits.
#define CONV2D_TC_WIN_VARIANTS(X)       \
    X(0, 64, 4, 3, 48, 2, false, 0)     \
    X(1, 64, 6, 2, 48, 2, false, 0)     \
    X(2, 128, 2, 3, 48, 2, false, 0)    \
    X(3, 128, 3, 2, 48, 2, false, 0)    \
    X(4, 256, 1, 3, 48, 2, false, 0)    \
    X(5, 64, 4, 4, 32, 2, false, 0)     \
    X(6, 128, 2, 4, 32, 2, false, 0)    \
    X(7, 64, 1, 1, 32, 4, true, 72)     \
    X(8, 128, 1, 1, 32, 4, true, 72)    \
    X(9, 128, 3, 3, 25, 2, false, 0)    \
    X(10, 128, 3, 3, 33, 2, false, 0)

template <typename T>
conv2d_status_t dispatch_window(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
#define CONV2D_TC_WCASE(vid, vbn, vks, vst, vwk, vnw, vres, vrk) \
    if (pl.tc.win_variant == vid) return launch_tc_window<T, vbn, vks, vst, vwk, vnw, vres, vrk>(s, pl, t, st);
    CONV2D_TC_WIN_VARIANTS(CONV2D_TC_WCASE)
#undef CONV2D_TC_WCASE
    return CONV2D_ERR_INTERNAL;
}

template <typename T, bool A_TILE>
conv2d_status_t dispatch_bn(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st) {
    if (pl.tc.cta2) {
#define CONV2D_TC_C2CASE(vbn, vks, vst) \
    if (pl.tc.BN == vbn && pl.tc.ksub == vks) return launch_tc<T, vbn, vks, vst, A_TILE, true>(s, pl, t, st);
        CONV2D_TC_CTA2_VARIANTS(CONV2D_TC_C2CASE)
#undef CONV2D_TC_C2CASE
        return CONV2D_ERR_INTERNAL;
    }
#define CONV2D_TC_CASE(vbn, vks, vst) \
    if (pl.tc.BN == vbn && pl.tc.ksub == vks) return launch_tc<T, vbn, vks, vst, A_TILE, false>(s, pl, t, st);
    CONV2D_TC_VARIANTS(CONV2D_TC_CASE)
#undef CONV2D_TC_CASE
    return CONV2D_ERR_INTERNAL;
}

// 1x1, stride 1, no padding: output pixel m reads input pixel m.
bool plain_matrix_a(const Shape &s) {
    return s.R == 1 && s.S == 1 && s.stride == 1 && s.pad == 0;
}

}  // namespace

bool tc_shape_ok(const Shape &s, const Tensors *t) {
    if (s.dtype != CONV2D_F16 && s.dtype != CONV2D_BF16) return false;
    if (s.layout != CONV2D_NHWC) return false;
    if (s.C % 8 != 0 || s.K % 8 != 0) return false;               // 16-byte rows for TMA and stores
    if (s.stride > 8) return false;                               // TMA traversal stride limit
    if (s.pad > 127) return false;                                // im2col corner range
    const int64_t up_h = (int64_t)s.pad - (int64_t)s.dil * (s.R - 1);
    const int64_t up_w = (int64_t)s.pad - (int64_t)s.dil * (s.S - 1);
    if (up_h < -128 || up_w < -128 || up_h > 127 || up_w > 127) return false;
    if ((int64_t)s.dil * (s.R - 1) > 255 || (int64_t)s.dil * (s.S - 1) > 255) return false;
    if ((int64_t)s.N * s.H * s.W >= ((int64_t)1 << 31)) return false;
    if (s.M >= ((int64_t)1 << 31) - 256) return false;   // row coordinates of the y map are 32-bit
    if (t) {
        auto a16 = [](const void *q) { return ((uintptr_t)q & 15) == 0; };
        if (!a16(t->x) || !a16(t->w) || !a16(t->y)) return false;
    }
    return true;
}

size_t tc_smem_bytes(const TcTile &t) {
    if (t.cta2) {
#define CONV2D_TC_C2SMEM(vbn, vks, vst) \
    if (t.BN == vbn && t.ksub == vks) return TcSmem<vbn, vks, vst, true>::kBytes;
        CONV2D_TC_CTA2_VARIANTS(CONV2D_TC_C2SMEM)
#undef CONV2D_TC_C2SMEM
        return (size_t)1 << 30;
    }
#define CONV2D_TC_SMEM(vbn, vks, vst) \
    if (t.BN == vbn && t.ksub == vks) return TcSmem<vbn, vks, vst>::kBytes;
    CONV2D_TC_VARIANTS(CONV2D_TC_SMEM)
#undef CONV2D_TC_SMEM
    return (size_t)1 << 30;
}

size_t tc_window_smem_bytes(const TcTile &t) {
#define CONV2D_TC_WSMEM(vid, vbn, vks, vst, vwk, vnw, vres, vrk) \
    if (t.win_variant == vid) return TcWinSmem<vbn, vks, vst, vwk, vnw, vres, vrk>::kBytes;
    CONV2D_TC_WIN_VARIANTS(CONV2D_TC_WSMEM)
#undef CONV2D_TC_WSMEM
    return (size_t)1 << 30;
}

int tc_window_variants() {
    int n = 0;
#define CONV2D_TC_WCOUNT(vid, vbn, vks, vst, vwk, vnw, vres, vrk) ++n;
    CONV2D_TC_WIN_VARIANTS(CONV2D_TC_WCOUNT)
#undef CONV2D_TC_WCOUNT
    return n;
}

TcWinVariant tc_window_variant(int id) {
    TcWinVariant v{};
#define CONV2D_TC_WGET(vid, vbn, vks, vst, vwk, vnw, vres, vrk) \
    if (id == vid) v = TcWinVariant{vbn, vks, vst, vwk, vnw, vres, vrk};
    CONV2D_TC_WIN_VARIANTS(CONV2D_TC_WGET)
#undef CONV2D_TC_WGET
    return v;
}

// Geometry checks of one window variant for a layer: the shifted window must
// fit its slot; resident weights need one output-channel tile and must fit.
bool tc_window_variant_ok(const Shape &s, int id) {
    const TcWinVariant v = tc_window_variant(id);
    if (v.bn == 0) return false;
    const WinGeom g = win_geom(s);
    if (g.max_shift + kBM > v.win_kb * 1024 / 128) return false;
    if (v.resident) {
        if (s.K > v.bn) return false;
        const int64_t cb = (s.C + kBK - 1) / kBK;
        if (cb * s.R * s.S * v.bn * kBK * 2 > (int64_t)v.res_kb * 1024) return false;
        if ((int64_t)s.R * s.S > 256) return false;   // box dimension limit
    }
    return true;
}

// Window mode needs stride 1, padded rows of at most 128 pixels, and the
// shifted window (largest tap shift + 128 rows) inside one window slot.
bool tc_window_ok(const Shape &s) {
    if (s.stride != 1) return false;
    const WinGeom g = win_geom(s);
    if (g.Wp > kBM || g.TR < 1) return false;
    if (g.TRW > 256) return false;
    if (g.max_shift + kBM > 48 * 1024 / 128) return false;
    return true;
}

int tc_num_variants() {
    int n = 0;
#define CONV2D_TC_COUNT(vbn, vks, vst) ++n;
    CONV2D_TC_VARIANTS(CONV2D_TC_COUNT)
#undef CONV2D_TC_COUNT
    return n;
}

int tc_cta2_num_variants() {
    int n = 0;
#define CONV2D_TC_C2COUNT(vbn, vks, vst) ++n;
    CONV2D_TC_CTA2_VARIANTS(CONV2D_TC_C2COUNT)
#undef CONV2D_TC_C2COUNT
    return n;
}

int tc_stages(int bn, int ksub) {
#define CONV2D_TC_ST(vbn, vks, vst) \
    if (bn == vbn && ksub == vks) return vst;
    CONV2D_TC_VARIANTS(CONV2D_TC_ST)
#undef CONV2D_TC_ST
    return 0;
}

int tc_cta2_stages(int bn, int ksub) {
#define CONV2D_TC_C2ST(vbn, vks, vst) \
    if (bn == vbn && ksub == vks) return vst;
    CONV2D_TC_CTA2_VARIANTS(CONV2D_TC_C2ST)
#undef CONV2D_TC_C2ST
    return 0;
}

conv2d_status_t tc_launch(const Shape &s, const Plan &p, const Tensors &t, cudaStream_t st) {
    if (p.tc.window) {
        if (!tc_window_ok(s)) return CONV2D_ERR_INTERNAL;
        if (s.dtype == CONV2D_BF16) return dispatch_window<__nv_bfloat16>(s, p, t, st);
        return dispatch_window<__half>(s, p, t, st);
    }
    const bool a_tile = plain_matrix_a(s) && !p.tc.force_im2col;
    if (s.dtype == CONV2D_BF16)
        return a_tile ? dispatch_bn<__nv_bfloat16, true>(s, p, t, st)
                      : dispatch_bn<__nv_bfloat16, false>(s, p, t, st);
    return a_tile ? dispatch_bn<__half, true>(s, p, t, st) : dispatch_bn<__half, false>(s, p, t, st);
}

}  // namespace conv2d

#ifdef CONV2D_TC_TRACE
extern "C" int conv2d_tc_trace_dump(unsigned long long *out, unsigned int *counts) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(counts, conv2d::g_tc_trace_n, sizeof(unsigned int) * 4) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(out, conv2d::g_tc_trace, sizeof(unsigned long long) * 4 * 8192) != cudaSuccess)
        return -1;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(conv2d::g_tc_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif
